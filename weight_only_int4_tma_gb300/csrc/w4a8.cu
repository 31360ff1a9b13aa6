// W4A8 path (LiquidQuant): 4-bit weight codes turned back into int8 inside the kernel,
// multiplied with per-row int8 activations, summed exactly and scaled in fp32.  Source:
// "W4A8量化计算优化：提升LLM推理效率的关键技术" §2.1 (the congruence
// Q_i8 = (Q_u4 * s_u8 + a) XOR 0x80 with an integer step s_u8 <= 16, so that one IMAD
// dequantises four codes packed one per byte), §3.1-3.2 (dequantise in registers and
// feed the multiply directly; the int8 weights are never written back).
//
// The page feeds an int8 x int8 -> int32 tensor-core MMA.  On sm_103a the int8 MMA of
// the tcgen05 family does not exist (ptxas rejects kind::i8 for this target), and the
// int8 mma.sync runs at about the rate of dp4a on the CUDA cores (measured 75 and 72
// T MAC/s), while the f16 mma.sync runs at 297 T MAC/s.  Every int8 value is exact in
// fp16, and one 128-K block's partial sum of int8 products stays below 2^24 in
// magnitude (128 * 127 * 128), so an f16 MMA with fp32 accumulation computes each
// block's integer sum exactly; the blocks' sums are then added in int32.  The GEMM
// therefore takes the f16 mma.sync for 3..16 activation rows and dp4a for one or two
// rows (where the MMA's fixed 8-row width would waste most of its work).  Either way
// the result is the exact integer sum, the same bits as the plain definition.
//
// Packed blob (private to this file, versioned by its header):
//   [0, 128)            header (W4A8Header)
//   blocks              one per (16-channel tile t, 128-K block kb), tiles in order,
//                       blocks of one tile contiguous along K; kW4a8BlockBytes each:
//     [0, 1024)         codes in the mma.sync fragment order: lane l = 4g + i (g = l / 4,
//                       i = l % 4) owns 32 bytes at 32 l, one word per MMA step j; byte b
//                       of word j holds the codes of K value 32 i + 4 j + b of channel g
//                       (low nibble) and of channel g + 8 (high nibble).  So
//                       (x & 0x0F0F0F0F) and ((x >> 4) & 0x0F0F0F0F) are four codes of
//                       one channel in K order, a lane's eight words cover 32 consecutive
//                       K values (the activations it needs are 32 contiguous bytes per
//                       row), and a warp reads a block as 1 KB of contiguous 32-byte
//                       pieces.
//     [1024, 1056)      word g: step and offset of channel g (bytes 0, 1) and of
//                       channel g + 8 (bytes 2, 3).
//   s_w                 fp32 [Np], the per-channel scale (0 past N).
// N is padded to Np = a multiple of 16 (padded channels: codes 0, step 1, offset 128, so
// their int8 weights are exactly 0); K must be a multiple of 128 (one group per block).
//
// In MMA step j the MMA's K index k' = 2i + e (e = 0, 1) stands for K value 32i + 4j + e
// and k' = 8 + 2i + e for 32i + 4j + 2 + e, for the weights and the activations alike; a
// sum over K does not depend on the order of its terms, and these sums are exact.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "launch.h"
#include "ptx.cuh"

namespace w4g {

namespace {

constexpr uint32_t kW4a8Magic = 0x38413457u;  // "W4A8"
constexpr uint32_t kW4a8Version = 2;
constexpr int kW4a8Group = 128;
constexpr int kW4a8TileN = 16;
constexpr uint32_t kW4a8CodeBytes = kW4a8TileN * kW4a8Group / 2;             // 1024
constexpr uint32_t kW4a8BlockBytes = kW4a8CodeBytes + 2 * kW4a8TileN;        // 1056
constexpr int kW4a8Threads = 256;
constexpr int kW4a8Warps = kW4a8Threads / 32;  // K slots of a GEMM CTA
constexpr int kStatusInvalidArg = -1;          // w4a16_status W4A16_ERR_INVALID_ARG

struct W4A8Header {
    uint32_t magic;
    uint32_t version;
    int32_t N;
    int32_t K;
    uint32_t block_bytes;
    uint32_t reserved0;
    uint64_t body_offset;
    uint64_t sw_offset;
    uint64_t total_bytes;
    uint32_t reserved[20];
};
static_assert(sizeof(W4A8Header) == 128, "header must be 128 bytes");

__host__ __device__ constexpr int w4a8_tiles(int N) { return (N + kW4a8TileN - 1) / kW4a8TileN; }

__host__ __device__ inline uint64_t w4a8_sw_offset(int N, int K) {
    return 128ull + static_cast<uint64_t>(w4a8_tiles(N)) * (K / kW4a8Group) * kW4a8BlockBytes;
}

// Four codes (one per byte, each 0..15) -> code * s + a per byte, i.e. the int8 weights
// plus 128 (the congruence before its XOR): the products code * s stay below 256 and,
// with the offset added, every byte stays at most 255 (the format's precondition), so
// no carry crosses a byte.
__device__ __forceinline__ uint32_t biased_i8x4(uint32_t codes, uint32_t s, uint32_t add) {
    return codes * s + add;
}

__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t ld_stream_u32(const void* p) {
    uint32_t v;
    asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

// ---- repack ------------------------------------------------------------------------

// One CTA per (tile, block); thread (j, l) = (tid / 32, tid % 32) writes word j of lane
// l: the codes of K values 32 i + 4 j + (0..3) of channels g and g + 8 (g = l / 4,
// i = l % 4).  Lanes 4g of step 0 also write the step and offset word g, and in block 0
// of the tile the two channels' s_w.  Codes whose byte value code * s + a would pass
// 255, and steps outside 1..16, are recorded as W4A16_ERR_INVALID_ARG in the status word
// (the blob is written anyway).
__global__ void __launch_bounds__(256) w4a8_repack_kernel(
    const uint32_t* __restrict__ qweight, const uint8_t* __restrict__ s_u8,
    const uint8_t* __restrict__ off, const float* __restrict__ s_w, int N, int K,
    uint8_t* __restrict__ packed, int* status) {
    const int kblocks = K / kW4a8Group;
    const int t = static_cast<int>(blockIdx.x) / kblocks;
    const int kb = static_cast<int>(blockIdx.x) - t * kblocks;
    const int j = static_cast<int>(threadIdx.x) >> 5;
    const int l = static_cast<int>(threadIdx.x) & 31;
    const int g = l >> 2, i = l & 3;
    uint8_t* blk = packed + 128 + static_cast<size_t>(blockIdx.x) * kW4a8BlockBytes;
    const int k0 = kb * kW4a8Group + 32 * i + 4 * j;  // first of the four K values
    uint32_t codes[2], sv[2], av[2];
    bool bad = false;
#pragma unroll
    for (int h = 0; h < 2; ++h) {  // channel g (h = 0) and g + 8 (h = 1)
        const int n = t * kW4a8TileN + g + 8 * h;
        uint32_t s = 1, a = 128, c = 0;
        if (n < N) {
            s = s_u8[static_cast<size_t>(n) * kblocks + kb];
            a = off[static_cast<size_t>(n) * kblocks + kb];
            const uint32_t w = qweight[static_cast<size_t>(n) * (K / 8) + k0 / 8];
            c = (w >> (4 * (k0 & 7))) & 0xFFFFu;  // four nibbles, K order
        }
        bad |= s < 1 || s > 16;
#pragma unroll
        for (int b = 0; b < 4; ++b) bad |= ((c >> (4 * b)) & 0xFu) * s + a > 255u;
        codes[h] = c;
        sv[h] = s;
        av[h] = a;
    }
    if (bad) record_status(status, kStatusInvalidArg);
    uint32_t word = 0;
#pragma unroll
    for (int b = 0; b < 4; ++b)
        word |= (((codes[0] >> (4 * b)) & 0xFu) | (((codes[1] >> (4 * b)) & 0xFu) << 4)) << (8 * b);
    *reinterpret_cast<uint32_t*>(blk + 32 * l + 4 * j) = word;
    if (j == 0 && i == 0) {
        *reinterpret_cast<uint32_t*>(blk + kW4a8CodeBytes + 4 * g) =
            sv[0] | (av[0] << 8) | (sv[1] << 16) | (av[1] << 24);
        if (kb == 0) {
            float* sw = reinterpret_cast<float*>(packed + w4a8_sw_offset(N, K));
            const int n0 = t * kW4a8TileN + g;
            sw[n0] = n0 < N ? s_w[n0] : 0.0f;
            sw[n0 + 8] = n0 + 8 < N ? s_w[n0 + 8] : 0.0f;
        }
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        W4A8Header h{};
        h.magic = kW4a8Magic;
        h.version = kW4a8Version;
        h.N = N;
        h.K = K;
        h.block_bytes = kW4a8BlockBytes;
        h.body_offset = 128;
        h.sw_offset = w4a8_sw_offset(N, K);
        h.total_bytes = h.sw_offset + 4ull * w4a8_tiles(N) * kW4a8TileN;
        *reinterpret_cast<W4A8Header*>(packed) = h;
    }
}

// A later kernel launched with programmatic dependent launch may start while this one
// still runs; this empty kernel keeps it from overlapping the repack itself.
__global__ void w4a8_fence_kernel() {}

__device__ __forceinline__ bool w4a8_header_ok(const uint8_t* packed, int N, int K) {
    const W4A8Header* h = reinterpret_cast<const W4A8Header*>(packed);
    return h->magic == kW4a8Magic && h->version == kW4a8Version && h->N == N && h->K == K &&
           h->block_bytes == kW4a8BlockBytes && h->body_offset == 128 &&
           h->sw_offset == w4a8_sw_offset(N, K);
}

// ---- debug dequant: the int8 weights W_i8[N][K] the GEMM multiplies -------------------

// Thread (j, l) of a block's CTA expands word j of lane l with the GEMM's arithmetic
// (one IMAD per four codes, then the XOR) into the four int8 weights of channels g and
// g + 8.
__global__ void __launch_bounds__(256) w4a8_dequant_debug_kernel(
    const uint8_t* __restrict__ packed, int N, int K, int8_t* __restrict__ W, int* status) {
    __shared__ int ok;
    if (threadIdx.x == 0) {
        ok = w4a8_header_ok(packed, N, K);
        if (!ok && blockIdx.x == 0) record_status(status, kStatusFormat);
    }
    __syncthreads();
    if (!ok) return;
    const int kblocks = K / kW4a8Group;
    const int t = static_cast<int>(blockIdx.x) / kblocks;
    const int kb = static_cast<int>(blockIdx.x) - t * kblocks;
    const int j = static_cast<int>(threadIdx.x) >> 5;
    const int l = static_cast<int>(threadIdx.x) & 31;
    const int g = l >> 2, i = l & 3;
    const uint8_t* blk = packed + 128 + static_cast<size_t>(blockIdx.x) * kW4a8BlockBytes;
    const uint32_t x = *reinterpret_cast<const uint32_t*>(blk + 32 * l + 4 * j);
    const uint32_t meta = *reinterpret_cast<const uint32_t*>(blk + kW4a8CodeBytes + 4 * g);
    const uint32_t w0 = biased_i8x4(x & 0x0F0F0F0Fu, meta & 0xFFu,
                                    ((meta >> 8) & 0xFFu) * 0x01010101u) ^ 0x80808080u;
    const uint32_t w1 = biased_i8x4((x >> 4) & 0x0F0F0F0Fu, (meta >> 16) & 0xFFu,
                                    (meta >> 24) * 0x01010101u) ^ 0x80808080u;
    const int k0 = kb * kW4a8Group + 32 * i + 4 * j;
    const int n0 = t * kW4a8TileN + g;
    if (n0 < N) *reinterpret_cast<uint32_t*>(W + static_cast<size_t>(n0) * K + k0) = w0;
    if (n0 + 8 < N) *reinterpret_cast<uint32_t*>(W + static_cast<size_t>(n0 + 8) * K + k0) = w1;
}

// ---- per-row int8 activations ------------------------------------------------------

template <int DT>
__device__ __forceinline__ float dtype_bits_to_f32(uint32_t b) {
    if constexpr (DT == 0) return __half2float(__ushort_as_half(static_cast<unsigned short>(b)));
    else return __bfloat162float(__ushort_as_bfloat16(static_cast<unsigned short>(b)));
}

// One thread-block cluster of kQuantCluster CTAs per row m, each CTA a slice of K/8
// values: amax = max |A[m, :]| (exact; the CTAs' partial maxima are combined through
// distributed shared memory), s_a = amax / 127 (1 for an all-zero row), A_i8 = rint(A /
// s_a) clipped to [-127, 127]; division and rounding in fp32, round to nearest even, as
// the oracle states them.  A slice is at most kQuantThreads * kQuantVec 16-byte pieces
// (K <= 131072), read once into registers with every load issued before the first use.
constexpr int kQuantCluster = 8;
constexpr int kQuantThreads = 256;
constexpr int kQuantVec = 8;  // 16-byte pieces per thread held in registers

template <int DT>
__device__ __forceinline__ float amax_piece(uint4 v, float amax) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        amax = fmaxf(amax, fabsf(dtype_bits_to_f32<DT>(w[j] & 0xFFFFu)));
        amax = fmaxf(amax, fabsf(dtype_bits_to_f32<DT>(w[j] >> 16)));
    }
    return amax;
}

template <int DT>
__device__ __forceinline__ uint2 quantize_piece(uint4 v, float s) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[2] = {0, 0};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const uint32_t bits = (w[j >> 1] >> (16 * (j & 1))) & 0xFFFFu;
        int q = __float2int_rn(__fdiv_rn(dtype_bits_to_f32<DT>(bits), s));
        q = max(-127, min(127, q));
        o[j >> 2] |= (static_cast<uint32_t>(q) & 0xFFu) << (8 * (j & 3));
    }
    return make_uint2(o[0], o[1]);
}

template <int DT>
__global__ void __launch_bounds__(kQuantThreads) w4a8_quantize_kernel(
    const uint16_t* __restrict__ A, int K, int8_t* __restrict__ A_i8, float* __restrict__ s_a) {
    __shared__ float wmax[kQuantThreads / 32];
    __shared__ float part;   // this CTA's maximum, read by the whole cluster
    __shared__ float s_row;
    grid_dep_wait();  // A belongs to the previous kernel until here
    const int m = static_cast<int>(blockIdx.x) / kQuantCluster;
    const uint32_t c = cluster_ctarank();
    const int tid = static_cast<int>(threadIdx.x);
    const int per = K / 8 / kQuantCluster;  // 16-byte pieces of this CTA's slice
    const uint4* row = reinterpret_cast<const uint4*>(A + static_cast<size_t>(m) * K) + c * per;
    uint2* out = reinterpret_cast<uint2*>(A_i8 + static_cast<size_t>(m) * K) + c * per;
    uint4 v[kQuantVec];
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < kQuantVec; ++j) {
        const int idx = tid + j * kQuantThreads;
        v[j] = idx < per ? __ldg(row + idx) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int j = 0; j < kQuantVec; ++j) amax = amax_piece<DT>(v[j], amax);
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, d));
    if ((tid & 31) == 0) wmax[tid >> 5] = amax;
    __syncthreads();
    if (tid == 0) {
        float mx = wmax[0];
        for (int w = 1; w < kQuantThreads / 32; ++w) mx = fmaxf(mx, wmax[w]);
        part = mx;
    }
    cluster_sync_all();  // every CTA's maximum is in place
    if (tid == 0) {
        float mx = 0.0f;
        for (uint32_t r = 0; r < kQuantCluster; ++r)
            mx = fmaxf(mx, ld_dsmem_f32(map_to_rank(smem_addr(&part), r)));
        const float s = mx > 0.0f ? __fdiv_rn(mx, 127.0f) : 1.0f;
        s_row = s;
        if (c == 0) s_a[m] = s;
    }
    cluster_sync_all();  // no CTA leaves while another may still read its maximum
    grid_dep_launch();
    const float s = s_row;
#pragma unroll
    for (int j = 0; j < kQuantVec; ++j) {
        const int idx = tid + j * kQuantThreads;
        if (idx < per) out[idx] = quantize_piece<DT>(v[j], s);
    }
}

// ---- the GEMM ----------------------------------------------------------------------

// Dynamic shared memory of a GEMM CTA: the warps' partials, 8 slots x 16 channels x MT
// rows of int32.
template <int MT>
constexpr uint32_t w4a8_smem_bytes() { return 512u * MT; }

// Two biased int8 values (bytes sel picks, each v + 128) -> their values as an fp16 pair:
// 0x6400 | byte is 1024 + byte exactly, and subtracting 1152 leaves v exactly.
__device__ __forceinline__ uint32_t biased_u8x2_to_f16x2(uint32_t u, uint32_t sel) {
    uint32_t d = __byte_perm(u, 0x64646464u, sel);
    asm("sub.rn.f16x2 %0, %0, %1;" : "+r"(d) : "r"(0x64806480u));
    return d;
}

__device__ __forceinline__ void mma_f16_16x8x16(float (&d)[4], uint32_t a0, uint32_t a1,
                                                uint32_t a2, uint32_t a3, uint32_t b0,
                                                uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// One 128-K block of this lane's two channels (g and g + 8) with MT <= 2 activation rows,
// by dp4a: acc[h][m] += the int8 products of channel g + 8h with row m over the lane's
// four K values of each step j; xa[m][j]: those four activations of row m.
template <int MT>
__device__ __forceinline__ void w4a8_block_dp4a(const uint4 (&w)[2], uint32_t meta,
                                                const uint32_t (&xa)[MT][8], int (&acc)[2][MT]) {
    const uint32_t s0 = meta & 0xFFu, add0 = ((meta >> 8) & 0xFFu) * 0x01010101u;
    const uint32_t s1 = (meta >> 16) & 0xFFu, add1 = (meta >> 24) * 0x01010101u;
    const uint32_t x[8] = {w[0].x, w[0].y, w[0].z, w[0].w, w[1].x, w[1].y, w[1].z, w[1].w};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int w0 = static_cast<int>(biased_i8x4(x[j] & 0x0F0F0F0Fu, s0, add0) ^ 0x80808080u);
        const int w1 = static_cast<int>(biased_i8x4((x[j] >> 4) & 0x0F0F0F0Fu, s1, add1) ^ 0x80808080u);
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            acc[0][m] = __dp4a(w0, static_cast<int>(xa[m][j]), acc[0][m]);
            acc[1][m] = __dp4a(w1, static_cast<int>(xa[m][j]), acc[1][m]);
        }
    }
}

// One 128-K block of the warp's 16 channels with NT groups of 8 activation rows, by f16
// mma.sync (m16n8k16): the weights, as int8 values in fp16, are the A fragments (rows g
// and g + 8 of the tile), the activations the B fragments (row 8t + g of group t; xa[t][j]
// holds its four int8 values at this lane's K offset of step j).  The block's sums are
// accumulated in fp32 from zero (exact: every partial sum is an integer below 2^24) and
// then added to iacc in int32.
template <int NT>
__device__ __forceinline__ void w4a8_block_mma(const uint4 (&w)[2], uint32_t meta,
                                               const uint32_t (&xa)[NT][8], int (&iacc)[NT][4]) {
    const uint32_t s0 = meta & 0xFFu, add0 = ((meta >> 8) & 0xFFu) * 0x01010101u;
    const uint32_t s1 = (meta >> 16) & 0xFFu, add1 = (meta >> 24) * 0x01010101u;
    const uint32_t x[8] = {w[0].x, w[0].y, w[0].z, w[0].w, w[1].x, w[1].y, w[1].z, w[1].w};
    float f[NT][4];
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
        for (int e = 0; e < 4; ++e) f[t][e] = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const uint32_t u0 = biased_i8x4(x[j] & 0x0F0F0F0Fu, s0, add0);
        const uint32_t u1 = biased_i8x4((x[j] >> 4) & 0x0F0F0F0Fu, s1, add1);
        const uint32_t a0 = biased_u8x2_to_f16x2(u0, 0x4140u);  // channel g, K 4i, 4i+1
        const uint32_t a2 = biased_u8x2_to_f16x2(u0, 0x4342u);  // channel g, K 4i+2, 4i+3
        const uint32_t a1 = biased_u8x2_to_f16x2(u1, 0x4140u);  // channel g + 8
        const uint32_t a3 = biased_u8x2_to_f16x2(u1, 0x4342u);
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            const uint32_t av = xa[t][j] ^ 0x80808080u;
            mma_f16_16x8x16(f[t], a0, a1, a2, a3, biased_u8x2_to_f16x2(av, 0x4140u),
                            biased_u8x2_to_f16x2(av, 0x4342u));
        }
    }
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
        for (int e = 0; e < 4; ++e) iacc[t][e] += __float2int_rn(f[t][e]);
}

template <int DT>
__device__ __forceinline__ uint16_t w4a8_f32_to_dtype(float v) {
    if constexpr (DT == 0) return __half_as_ushort(__float2half_rn(v));
    else return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

// Work split.  A CTA owns one 16-channel tile over the whole K range; its 8 warps are K
// slots taking the 128-K blocks slot, slot + 8, ...  Each lane keeps the codes (32
// bytes) of two blocks in flight in registers: the loads for block b + 2 are issued as
// soon as block b is multiplied.  The activation words a lane needs travel the same way,
// read through L1, two blocks ahead (one for 16 rows, to keep three CTAs on an SM).  MT
// is 1 or 2 (dp4a) or 8 or 16 (f16 mma.sync, one or two groups of 8 rows).  The warps'
// int32 partials are summed in shared memory (exact, so the order does not matter).
// Epilogue per output element: fp32(acc) * s_a[m] * s_w[n], two fp32 multiplies rounded
// to nearest even, then one rounding to the output dtype.
template <int MT, int DT>
__global__ void __launch_bounds__(kW4a8Threads, MT == 16 ? 3 : 4) w4a8_gemm_kernel(
    const int8_t* __restrict__ A_i8, const float* __restrict__ s_a,
    const uint8_t* __restrict__ packed, uint16_t* __restrict__ Y, int* status, int M, int N,
    int K) {
    constexpr bool kMma = MT >= 8;
    constexpr int NT = kMma ? MT / 8 : 1;
    extern __shared__ __align__(16) int red[];  // the warps' partials, after the main loop
    __shared__ int s_ok;
    const int tid = static_cast<int>(threadIdx.x);
    const int slot = tid >> 5, l = tid & 31;
    const int g = l >> 2, i = l & 3;
    const int tile = static_cast<int>(blockIdx.x);

    if (tid == 0) {
        const int ok = w4a8_header_ok(packed, N, K);
        s_ok = ok;
        if (!ok && blockIdx.x == 0) record_status(status, kStatusFormat);
    }
    __syncthreads();
    if (!s_ok) return;
    if (tid == 0) grid_dep_launch();

    const int kblocks = K / kW4a8Group;
    const uint8_t* tile_p = packed + 128 + static_cast<size_t>(tile) * kblocks * kW4a8BlockBytes;
    auto load = [&](int kb, uint4 (&w)[2], uint32_t& meta) {
        const uint8_t* blk = tile_p + static_cast<size_t>(kb) * kW4a8BlockBytes;
        w[0] = ld_stream_v4(blk + 32 * l);
        w[1] = ld_stream_v4(blk + 32 * l + 16);
        meta = ld_stream_u32(blk + kW4a8CodeBytes + 4 * g);
    };
    int acc[2][kMma ? 1 : MT];   // dp4a: channel g + 8h, row m
    int iacc[NT][4];             // mma: D fragment of group t
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int m = 0; m < (kMma ? 1 : MT); ++m) acc[h][m] = 0;
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
        for (int e = 0; e < 4; ++e) iacc[t][e] = 0;
    uint4 wa[2], wb[2];
    uint32_t ma = 0, mb = 0;
    // The packed weights do not depend on the previous kernel: the codes of the first two
    // blocks are requested before the dependency wait.
    if (slot < kblocks) load(slot, wa, ma);
    if (slot + kW4a8Warps < kblocks) load(slot + kW4a8Warps, wb, mb);
    grid_dep_wait();  // A_i8 and s_a (and Y) belong to the previous kernel until here
    {
        // Each lane loads the activation words its blocks need -- K values 32i .. 32i + 31
        // of row r (dp4a: every row; MMA: row 8t + g of group t) -- from global memory,
        // L1-cached (every CTA reads the same rows), ahead of the block that uses them;
        // rows past M read as zero.  The warps of a CTA run independently until the final
        // reduction.
        constexpr int R = kMma ? NT : MT;
        uint32_t xa[R][8], xb[(R <= 1 || !kMma) ? R : 1][8];
        auto load_a = [&](int kb, uint32_t (&xr)[R][8]) {
#pragma unroll
            for (int q = 0; q < R; ++q) {
                const int row = kMma ? 8 * q + g : q;
                uint4 lo = make_uint4(0, 0, 0, 0), hi = lo;
                if (row < M) {
                    const uint4* p = reinterpret_cast<const uint4*>(
                        A_i8 + static_cast<size_t>(row) * K + kb * kW4a8Group + 32 * i);
                    lo = __ldg(p);
                    hi = __ldg(p + 1);
                }
                xr[q][0] = lo.x; xr[q][1] = lo.y; xr[q][2] = lo.z; xr[q][3] = lo.w;
                xr[q][4] = hi.x; xr[q][5] = hi.y; xr[q][6] = hi.z; xr[q][7] = hi.w;
            }
        };
        auto block = [&](const uint4 (&w)[2], uint32_t meta, const uint32_t (&xr)[R][8]) {
            if constexpr (kMma) w4a8_block_mma<NT>(w, meta, xr, iacc);
            else w4a8_block_dp4a<MT>(w, meta, xr, acc);
        };
        if constexpr (R <= 1 || !kMma) {
            // activations two blocks ahead, like the codes
            if (slot < kblocks) load_a(slot, xa);
            if (slot + kW4a8Warps < kblocks) load_a(slot + kW4a8Warps, xb);
            for (int kb = slot; kb < kblocks; kb += 2 * kW4a8Warps) {
                block(wa, ma, xa);
                if (kb + 2 * kW4a8Warps < kblocks) {
                    load(kb + 2 * kW4a8Warps, wa, ma);
                    load_a(kb + 2 * kW4a8Warps, xa);
                }
                if (kb + kW4a8Warps < kblocks) {
                    block(wb, mb, xb);
                    if (kb + 3 * kW4a8Warps < kblocks) {
                        load(kb + 3 * kW4a8Warps, wb, mb);
                        load_a(kb + 3 * kW4a8Warps, xb);
                    }
                }
            }
        } else {
            // 16 rows: activations one block ahead in one set of registers (a second set
            // would cost the CTA its third slot on an SM)
            if (slot < kblocks) load_a(slot, xa);
            for (int kb = slot; kb < kblocks; kb += 2 * kW4a8Warps) {
                block(wa, ma, xa);
                if (kb + kW4a8Warps < kblocks) load_a(kb + kW4a8Warps, xa);
                if (kb + 2 * kW4a8Warps < kblocks) load(kb + 2 * kW4a8Warps, wa, ma);
                if (kb + kW4a8Warps < kblocks) {
                    block(wb, mb, xa);
                    if (kb + 2 * kW4a8Warps < kblocks) load_a(kb + 2 * kW4a8Warps, xa);
                    if (kb + 3 * kW4a8Warps < kblocks) load(kb + 3 * kW4a8Warps, wb, mb);
                }
            }
        }
    }
    // The warps' partials: red[slot][channel][row].
    if constexpr (kMma) {
#pragma unroll
        for (int t = 0; t < NT; ++t)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                red[(slot * kW4a8TileN + g + 8 * (e >> 1)) * MT + 8 * t + 2 * i + (e & 1)] = iacc[t][e];
    } else {
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                int v = acc[h][m];  // the four lanes of a channel pair hold K quarters
                v += __shfl_xor_sync(0xFFFFFFFFu, v, 1);
                v += __shfl_xor_sync(0xFFFFFFFFu, v, 2);
                if (i == 0) red[(slot * kW4a8TileN + g + 8 * h) * MT + m] = v;
            }
    }
    __syncthreads();
    const float* sw = reinterpret_cast<const float*>(packed + w4a8_sw_offset(N, K));
    for (int e = tid; e < kW4a8TileN * M; e += kW4a8Threads) {
        const int m = e / kW4a8TileN, row = e % kW4a8TileN;
        const int n = tile * kW4a8TileN + row;
        if (n < N) {
            int sum = 0;
#pragma unroll
            for (int q = 0; q < kW4a8Warps; ++q) sum += red[(q * kW4a8TileN + row) * MT + m];
            float y = __int2float_rn(sum);
            y = __fmul_rn(y, s_a[m]);
            y = __fmul_rn(y, sw[n]);
            Y[static_cast<size_t>(m) * N + n] = w4a8_f32_to_dtype<DT>(y);
        }
    }
}

template <int MT, int DT>
int launch_w4a8_instance(const DeviceCtx& ctx, const int8_t* A_i8, const float* s_a,
                         const void* packed, int M, int N, int K, void* Y, cudaStream_t stream) {
    auto kern = w4a8_gemm_kernel<MT, DT>;
    constexpr uint32_t smem = w4a8_smem_bytes<MT>();
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(w4a8_tiles(N)), 1, 1);
    cfg.blockDim = dim3(kW4a8Threads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, A_i8, s_a,
                                             static_cast<const uint8_t*>(packed),
                                             static_cast<uint16_t*>(Y), ctx.status, M, N, K);
    return e == cudaSuccess ? 0 : -3;
}

template <int MT>
int launch_w4a8_mt(const DeviceCtx& ctx, const int8_t* A_i8, const float* s_a,
                   const void* packed, int M, int N, int K, int dtype, void* Y,
                   cudaStream_t stream) {
    return dtype == 0 ? launch_w4a8_instance<MT, 0>(ctx, A_i8, s_a, packed, M, N, K, Y, stream)
                      : launch_w4a8_instance<MT, 1>(ctx, A_i8, s_a, packed, M, N, K, Y, stream);
}

}  // namespace

size_t w4a8_blob_bytes(int N, int K) {
    return static_cast<size_t>(w4a8_sw_offset(N, K)) + 4ull * w4a8_tiles(N) * kW4a8TileN;
}

int launch_w4a8_repack(const DeviceCtx& ctx, const uint32_t* qweight, const uint8_t* s_u8,
                       const uint8_t* off, const float* s_w, int N, int K, void* packed,
                       cudaStream_t stream) {
    const unsigned blocks = static_cast<unsigned>(w4a8_tiles(N) * (K / kW4a8Group));
    w4a8_repack_kernel<<<blocks, 256, 0, stream>>>(qweight, s_u8, off, s_w, N, K,
                                                    static_cast<uint8_t*>(packed), ctx.status);
    if (cudaGetLastError() != cudaSuccess) return -3;
    w4a8_fence_kernel<<<1, 32, 0, stream>>>();
    return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

int launch_w4a8_dequant_debug(const DeviceCtx& ctx, const void* packed, int N, int K,
                              void* W_out, cudaStream_t stream) {
    const unsigned blocks = static_cast<unsigned>(w4a8_tiles(N) * (K / kW4a8Group));
    w4a8_dequant_debug_kernel<<<blocks, 256, 0, stream>>>(
        static_cast<const uint8_t*>(packed), N, K, static_cast<int8_t*>(W_out), ctx.status);
    return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

int launch_w4a8_quantize(const DeviceCtx& ctx, const void* A, int M, int K, int dtype,
                         int8_t* A_i8, float* s_a, cudaStream_t stream) {
    (void)ctx;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(M) * kQuantCluster, 1, 1);
    cfg.blockDim = dim3(kQuantThreads, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = kQuantCluster;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    const uint16_t* a = static_cast<const uint16_t*>(A);
    const cudaError_t e =
        dtype == 0 ? cudaLaunchKernelEx(&cfg, w4a8_quantize_kernel<0>, a, K, A_i8, s_a)
                   : cudaLaunchKernelEx(&cfg, w4a8_quantize_kernel<1>, a, K, A_i8, s_a);
    return e == cudaSuccess ? 0 : -3;
}

int launch_w4a8_gemm(const DeviceCtx& ctx, const int8_t* A_i8, const float* s_a,
                     const void* packed, int M, int N, int K, int dtype, void* Y,
                     cudaStream_t stream) {
    // dp4a for one or two rows, the f16 MMA (groups of 8 rows) above
    if (M <= 1) return launch_w4a8_mt<1>(ctx, A_i8, s_a, packed, M, N, K, dtype, Y, stream);
    if (M <= 2) return launch_w4a8_mt<2>(ctx, A_i8, s_a, packed, M, N, K, dtype, Y, stream);
    if (M <= 8) return launch_w4a8_mt<8>(ctx, A_i8, s_a, packed, M, N, K, dtype, Y, stream);
    if (M <= 16) return launch_w4a8_mt<16>(ctx, A_i8, s_a, packed, M, N, K, dtype, Y, stream);
    return -2;
}

}  // namespace w4g
