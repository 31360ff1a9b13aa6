// W4A8 path (LiquidQuant): 4-bit weight codes turned back into int8 inside the kernel,
// multiplied with per-row int8 activations, accumulated exactly in int32 and scaled in
// fp32.  Source: "W4A8量化计算优化：提升LLM推理效率的关键技术" §2.1 (the congruence
// Q_i8 = (Q_u4 * s_u8 + a) XOR 0x80 with an integer step s_u8 <= 16, so that one IMAD
// and one XOR dequantise four weights packed one per byte), §3.1-3.2 (dequantise in
// registers, feed the multiply directly, never write the int8 weights back).
//
// The int8 tensor-core MMA the page feeds (tcgen05.mma.kind::i8) is not available on
// sm_103a (ptxas rejects the kind for this target), so the int8 dot products run on the
// CUDA cores as dp4a: four int8 x int8 products and their sum added to an int32 in one
// instruction.  Integer accumulation is exact, so the result does not depend on the
// order of the K sum and equals the plain definition bit for bit.
//
// Packed blob (private to this file, versioned by its header):
//   [0, 128)              header (W4A8Header)
//   blocks                one per (32-channel tile t, 128-K block kb), tiles in order,
//                         blocks of one tile contiguous along K; kW4a8BlockBytes each:
//     [0, 2048)           codes: piece p (32 K values) x channel r (32) x 16 bytes.  The
//                         16 bytes of (p, r) are four words; word i holds K values
//                         32p + 8i + (0..7) with K value j in byte j & 3, low nibble for
//                         j < 4, high nibble for j >= 4.  So (x & 0x0F0F0F0F) and
//                         ((x >> 4) & 0x0F0F0F0F) are four consecutive codes each, one
//                         per byte, in K order -- the byte order of an int8 activation
//                         word -- and a warp whose lanes are 32 channels reads piece p of
//                         a block as 512 contiguous bytes.
//     [2048, 2112)        channel r's step s_u8 (byte 2r) and offset a (byte 2r + 1).
//   s_w                   fp32 [Np], the per-channel scale (0 past N).
// N is padded to Np = a multiple of 32 (padded channels: codes 0, step 1, offset 128, so
// their int8 weights are exactly 0); K must be a multiple of 128 (one group per block).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "launch.h"
#include "ptx.cuh"

namespace w4g {

namespace {

constexpr uint32_t kW4a8Magic = 0x38413457u;  // "W4A8"
constexpr uint32_t kW4a8Version = 1;
constexpr int kW4a8Group = 128;
constexpr int kW4a8TileN = 32;
constexpr uint32_t kW4a8CodeBytes = kW4a8TileN * kW4a8Group / 2;             // 2048
constexpr uint32_t kW4a8BlockBytes = kW4a8CodeBytes + 2 * kW4a8TileN;        // 2112
constexpr int kW4a8Threads = 256;
constexpr int kW4a8Warps = kW4a8Threads / 32;
constexpr int kStatusInvalidArg = -1;  // w4a16_status W4A16_ERR_INVALID_ARG

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

// Four codes (one per byte, each 0..15) -> four int8 weights by the congruence: the
// products code * s stay below 256 and, with the offset added, every byte stays at most
// 255 (the format's precondition), so no carry crosses a byte.
__device__ __forceinline__ int congruence_i8x4(uint32_t codes, uint32_t s, uint32_t add) {
    return static_cast<int>((codes * s + add) ^ 0x80808080u);
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

// One CTA per (tile, block); thread (p, r) = (tid / 32, tid % 32) writes the 16 code
// bytes of piece p of channel r; warp 0 also writes the channel's step and offset.
// Codes whose byte value code * s + a would pass 255, and steps outside 1..16, are
// recorded as W4A16_ERR_INVALID_ARG in the status word (the blob is written anyway).
__global__ void __launch_bounds__(128) w4a8_repack_kernel(
    const uint32_t* __restrict__ qweight, const uint8_t* __restrict__ s_u8,
    const uint8_t* __restrict__ off, const float* __restrict__ s_w, int N, int K,
    uint8_t* __restrict__ packed, int* status) {
    const int kblocks = K / kW4a8Group;
    const int t = static_cast<int>(blockIdx.x) / kblocks;
    const int kb = static_cast<int>(blockIdx.x) - t * kblocks;
    const int p = static_cast<int>(threadIdx.x) >> 5;
    const int r = static_cast<int>(threadIdx.x) & 31;
    const int n = t * kW4a8TileN + r;
    uint8_t* blk = packed + 128 + static_cast<size_t>(blockIdx.x) * kW4a8BlockBytes;

    uint32_t s = 1, a = 128;
    uint4 in = make_uint4(0, 0, 0, 0);
    if (n < N) {
        s = s_u8[static_cast<size_t>(n) * kblocks + kb];
        a = off[static_cast<size_t>(n) * kblocks + kb];
        in = *reinterpret_cast<const uint4*>(qweight + static_cast<size_t>(n) * (K / 8) +
                                              kb * 16 + p * 4);
    }
    const uint32_t words[4] = {in.x, in.y, in.z, in.w};
    uint32_t out[4];
    bool bad = s < 1 || s > 16;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint32_t o = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint32_t q = (words[i] >> (4 * j)) & 0xFu;
            bad |= q * s + a > 255u;
            o |= q << (8 * (j & 3) + 4 * (j >> 2));
        }
        out[i] = o;
    }
    if (bad) record_status(status, kStatusInvalidArg);
    *reinterpret_cast<uint4*>(blk + p * 512 + r * 16) = make_uint4(out[0], out[1], out[2], out[3]);
    if (p == 0) {
        blk[kW4a8CodeBytes + 2 * r] = static_cast<uint8_t>(s);
        blk[kW4a8CodeBytes + 2 * r + 1] = static_cast<uint8_t>(a);
        if (kb == 0) {
            float* sw = reinterpret_cast<float*>(packed + w4a8_sw_offset(N, K));
            sw[n] = n < N ? s_w[n] : 0.0f;
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

__global__ void __launch_bounds__(128) w4a8_dequant_debug_kernel(
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
    const int p = static_cast<int>(threadIdx.x) >> 5;
    const int r = static_cast<int>(threadIdx.x) & 31;
    const int n = t * kW4a8TileN + r;
    if (n >= N) return;
    const uint8_t* blk = packed + 128 + static_cast<size_t>(blockIdx.x) * kW4a8BlockBytes;
    const uint4 v = *reinterpret_cast<const uint4*>(blk + p * 512 + r * 16);
    const uint32_t s = blk[kW4a8CodeBytes + 2 * r];
    const uint32_t add = blk[kW4a8CodeBytes + 2 * r + 1] * 0x01010101u;
    const uint32_t x[4] = {v.x, v.y, v.z, v.w};
    int o[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        o[2 * i] = congruence_i8x4(x[i] & 0x0F0F0F0Fu, s, add);
        o[2 * i + 1] = congruence_i8x4((x[i] >> 4) & 0x0F0F0F0Fu, s, add);
    }
    int4* dst = reinterpret_cast<int4*>(W + static_cast<size_t>(n) * K + kb * kW4a8Group + p * 32);
    dst[0] = make_int4(o[0], o[1], o[2], o[3]);
    dst[1] = make_int4(o[4], o[5], o[6], o[7]);
}

// ---- per-row int8 activations ------------------------------------------------------

template <int DT>
__device__ __forceinline__ float dtype_bits_to_f32(uint32_t b) {
    if constexpr (DT == 0) return __half2float(__ushort_as_half(static_cast<unsigned short>(b)));
    else return __bfloat162float(__ushort_as_bfloat16(static_cast<unsigned short>(b)));
}

// One CTA of kQuantThreads threads per row m: amax = max |A[m, :]| (exact), s_a =
// amax / 127 (1 for an all-zero row), A_i8 = rint(A / s_a) clipped to [-127, 127];
// division and rounding in fp32, round to nearest even, as the oracle states them.
// Rows of up to kQuantThreads * kQuantVec * 8 values are read once into registers (all
// loads issued before the first is used); longer rows are read twice.
constexpr int kQuantThreads = 512;
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
    __shared__ float s_row;
    grid_dep_wait();  // A belongs to the previous kernel until here
    const int m = static_cast<int>(blockIdx.x);
    const int tid = static_cast<int>(threadIdx.x);
    const uint4* row = reinterpret_cast<const uint4*>(A + static_cast<size_t>(m) * K);
    uint2* out = reinterpret_cast<uint2*>(A_i8 + static_cast<size_t>(m) * K);
    const int nv = K / 8;
    const bool in_regs = nv <= kQuantThreads * kQuantVec;
    uint4 v[kQuantVec];
    float amax = 0.0f;
    if (in_regs) {
#pragma unroll
        for (int j = 0; j < kQuantVec; ++j) {
            const int i = tid + j * kQuantThreads;
            v[j] = i < nv ? __ldg(row + i) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int j = 0; j < kQuantVec; ++j) amax = amax_piece<DT>(v[j], amax);
    } else {
        for (int i = tid; i < nv; i += kQuantThreads) amax = amax_piece<DT>(__ldg(row + i), amax);
    }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, d));
    if ((tid & 31) == 0) wmax[tid >> 5] = amax;
    __syncthreads();
    if (tid == 0) {
        float mx = wmax[0];
        for (int w = 1; w < kQuantThreads / 32; ++w) mx = fmaxf(mx, wmax[w]);
        const float s = mx > 0.0f ? __fdiv_rn(mx, 127.0f) : 1.0f;
        s_row = s;
        s_a[m] = s;
    }
    __syncthreads();
    grid_dep_launch();
    const float s = s_row;
    if (in_regs) {
#pragma unroll
        for (int j = 0; j < kQuantVec; ++j) {
            const int i = tid + j * kQuantThreads;
            if (i < nv) out[i] = quantize_piece<DT>(v[j], s);
        }
    } else {
        for (int i = tid; i < nv; i += kQuantThreads) out[i] = quantize_piece<DT>(__ldg(row + i), s);
    }
}

// ---- the GEMM ----------------------------------------------------------------------

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Accumulator chains per activation row: two independent dp4a chains where there are
// only one or two rows, one where the rows already give enough independent chains.
template <int MT>
constexpr int w4a8_chains() { return MT <= 2 ? 2 : 1; }

// acc[m][*] += the int8 products of one 128-K block of this thread's channel with the
// MT activation rows staged in shared memory (rows past M hold zeros).  w: the block's
// four 16-byte pieces; meta: step in bits 0..7, offset in bits 8..15; a_s: row 0 of the
// block's int8 activations, row m at + m * kRow bytes.
template <int MT, uint32_t kRow>
__device__ __forceinline__ void w4a8_block(const uint4 (&w)[4], uint32_t meta,
                                           const uint8_t* a_s,
                                           int (&acc)[MT][w4a8_chains<MT>()]) {
    constexpr int C = w4a8_chains<MT>();
    const uint32_t s = meta & 0xFFu;
    const uint32_t add = ((meta >> 8) & 0xFFu) * 0x01010101u;
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        const uint32_t x[4] = {w[p].x, w[p].y, w[p].z, w[p].w};
        int wq[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            wq[2 * i] = congruence_i8x4(x[i] & 0x0F0F0F0Fu, s, add);
            wq[2 * i + 1] = congruence_i8x4((x[i] >> 4) & 0x0F0F0F0Fu, s, add);
        }
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            const uint4* ap = reinterpret_cast<const uint4*>(a_s + m * kRow + 32 * p);
            const uint4 a0 = ap[0], a1 = ap[1];
            const uint32_t av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i)
                acc[m][i % C] = __dp4a(wq[i], static_cast<int>(av[i]), acc[m][i % C]);
        }
    }
}

template <int DT>
__device__ __forceinline__ uint16_t w4a8_f32_to_dtype(float v) {
    if constexpr (DT == 0) return __half_as_ushort(__float2half_rn(v));
    else return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

// Dynamic shared memory of one GEMM CTA: two buffers of int8 activations, each MT rows
// x (K slots x 128) values (the activations of one round of blocks).
__host__ __device__ constexpr uint32_t w4a8_smem_bytes(int MT, int ROWS) {
    return 2u * MT * (kW4a8Warps * (32 / ROWS)) * kW4a8Group;
}

// Work split.  A CTA owns ROWS (16 or 32) consecutive output channels over the whole K
// range: thread lane % ROWS is the channel, and the 256 / ROWS K slots (ROWS lanes each)
// take the 128-K blocks slot, slot + slots, ...: round r of the CTA is blocks
// r * slots .. r * slots + slots - 1, one per slot.  Each thread keeps the weights of
// two rounds in flight in registers (the loads of round r + 2 are issued as soon as
// round r is multiplied); the int8 activations of a round are staged in shared memory
// by the whole CTA with cp.async, one round ahead, so that the dp4a chains read them at
// shared-memory latency.  The slots' int32 partials are summed in shared memory; the
// sum is exact, so the slot order does not matter.  Epilogue per output element:
// fp32(acc) * s_a[m] * s_w[n], two fp32 multiplies rounded to nearest even, then one
// rounding to the output dtype.
template <int MT, int DT, int ROWS>
__global__ void __launch_bounds__(kW4a8Threads, MT == 1 ? 4 : (MT == 2 ? 3 : 2)) w4a8_gemm_kernel(
    const int8_t* __restrict__ A_i8, const float* __restrict__ s_a,
    const uint8_t* __restrict__ packed, uint16_t* __restrict__ Y, int* status, int M, int N,
    int K) {
    constexpr int kSub = 32 / ROWS;
    constexpr int kSlots = kW4a8Warps * kSub;
    constexpr int C = w4a8_chains<MT>();
    constexpr uint32_t kRow = kSlots * kW4a8Group;  // bytes of one activation row per round
    constexpr uint32_t kBuf = MT * kRow;
    extern __shared__ __align__(16) uint8_t a_smem[];
    __shared__ int s_ok;
    const int tid = static_cast<int>(threadIdx.x);
    const int lane = tid & 31;
    const int rl = lane % ROWS;
    const int slot = (tid >> 5) * kSub + lane / ROWS;
    const int n0 = static_cast<int>(blockIdx.x) * ROWS;
    const int r = n0 % kW4a8TileN + rl;  // channel within its 32-channel tile

    if (tid == 0) {
        const int ok = w4a8_header_ok(packed, N, K);
        s_ok = ok;
        if (!ok && blockIdx.x == 0) record_status(status, kStatusFormat);
    }
    __syncthreads();
    if (!s_ok) return;
    if (tid == 0) grid_dep_launch();

    const int kblocks = K / kW4a8Group;
    const int rounds = (kblocks + kSlots - 1) / kSlots;
    const uint8_t* tile = packed + 128 +
                          static_cast<size_t>(n0 / kW4a8TileN) * kblocks * kW4a8BlockBytes;
    auto load = [&](int kb, uint4 (&w)[4], uint32_t& meta) {
        const uint8_t* blk = tile + static_cast<size_t>(kb) * kW4a8BlockBytes;
#pragma unroll
        for (int p = 0; p < 4; ++p) w[p] = ld_stream_v4(blk + p * 512 + r * 16);
        meta = ld_stream_u32(blk + kW4a8CodeBytes + (r & ~1) * 2) >> ((r & 1) * 16);
    };
    const uint32_t smem = smem_addr(a_smem);
    // The activations of round rr into buffer rr & 1: rows m < M, 16 bytes per copy
    // (pieces past K, in the last round only, are skipped: no block reads them).
    auto stage = [&](int rr) {
        constexpr int kPieces = static_cast<int>(kRow / 16);
        const int k0 = rr * static_cast<int>(kRow);
        const uint32_t buf = smem + (rr & 1) * kBuf;
        for (int e = tid; e < M * kPieces; e += kW4a8Threads) {
            const int m = e / kPieces, c = e % kPieces;
            if (k0 + c * 16 < K)
                cp_async16(buf + m * kRow + c * 16, A_i8 + static_cast<size_t>(m) * K + k0 + c * 16);
        }
    };
    // Rows M..MT-1 of both buffers are zero for the whole kernel (every block multiplies
    // all MT rows; those products are 0 and their sums are never stored).
    for (int e = tid; e < (MT - M) * static_cast<int>(kRow / 16) * 2; e += kW4a8Threads) {
        const int per_buf = (MT - M) * static_cast<int>(kRow / 16);
        const int bsel = e / per_buf, rem = e % per_buf;
        const int m = M + rem / static_cast<int>(kRow / 16), c = rem % static_cast<int>(kRow / 16);
        *reinterpret_cast<uint4*>(a_smem + bsel * kBuf + m * kRow + c * 16) = make_uint4(0, 0, 0, 0);
    }

    int acc[MT][C];
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int c = 0; c < C; ++c) acc[m][c] = 0;
    uint4 wa[4], wb[4];
    uint32_t ma = 0, mb = 0;
    // The packed weights do not depend on the previous kernel: the first two rounds are
    // requested before the dependency wait.
    if (slot < kblocks) load(slot, wa, ma);
    if (slot + kSlots < kblocks) load(slot + kSlots, wb, mb);
    grid_dep_wait();  // A_i8 and s_a (and Y) belong to the previous kernel until here
    stage(0);
    cp_async_commit();
    for (int rr = 0; rr < rounds; ++rr) {
        if (rr + 1 < rounds) stage(rr + 1);
        cp_async_commit();      // (an empty group in the last round)
        cp_async_wait<1>();     // this thread's copies of round rr have landed ...
        __syncthreads();        // ... and every other thread's
        const int kb = rr * kSlots + slot;
        if (kb < kblocks) {
            const uint8_t* a_s = a_smem + (rr & 1) * kBuf + slot * kW4a8Group;
            if (rr & 1) {
                w4a8_block<MT, kRow>(wb, mb, a_s, acc);
                if (kb + 2 * kSlots < kblocks) load(kb + 2 * kSlots, wb, mb);
            } else {
                w4a8_block<MT, kRow>(wa, ma, a_s, acc);
                if (kb + 2 * kSlots < kblocks) load(kb + 2 * kSlots, wa, ma);
            }
        }
        __syncthreads();        // buffer rr & 1 is free for round rr + 2
    }
    cp_async_wait<0>();
    // The activation buffers are reused for the slots' partials: red[slot][m][channel].
    int* red = reinterpret_cast<int*>(a_smem);
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        int t = acc[m][0];
#pragma unroll
        for (int c = 1; c < C; ++c) t += acc[m][c];
        red[(slot * MT + m) * ROWS + rl] = t;
    }
    __syncthreads();
    const float* sw = reinterpret_cast<const float*>(packed + w4a8_sw_offset(N, K));
    for (int e = tid; e < MT * ROWS; e += kW4a8Threads) {
        const int m = e / ROWS, jr = e - (e / ROWS) * ROWS;
        const int n = n0 + jr;
        if (m < M && n < N) {
            int sum = 0;
#pragma unroll
            for (int q = 0; q < kSlots; ++q) sum += red[(q * MT + m) * ROWS + jr];
            float y = __int2float_rn(sum);
            y = __fmul_rn(y, s_a[m]);
            y = __fmul_rn(y, sw[n]);
            Y[static_cast<size_t>(m) * N + n] = w4a8_f32_to_dtype<DT>(y);
        }
    }
}

template <int MT, int DT, int ROWS>
int launch_w4a8_instance(const DeviceCtx& ctx, const int8_t* A_i8, const float* s_a,
                         const void* packed, int M, int N, int K, void* Y, cudaStream_t stream) {
    auto kern = w4a8_gemm_kernel<MT, DT, ROWS>;
    constexpr uint32_t smem = w4a8_smem_bytes(MT, ROWS);
    static int configured_device = -1;  // attribute set once per device and instance
    if (configured_device != ctx.device) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem)) != cudaSuccess)
            return -3;
        configured_device = ctx.device;
    }
    const int np = w4a8_tiles(N) * kW4a8TileN;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(np / ROWS), 1, 1);
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

// CTAs of one instance resident per SM (queried once per device).
template <int MT, int DT, int ROWS>
int w4a8_occupancy(const DeviceCtx& ctx) {
    static int device = -1, occ = 0;
    if (device != ctx.device) {
        auto kern = w4a8_gemm_kernel<MT, DT, ROWS>;
        constexpr uint32_t smem = w4a8_smem_bytes(MT, ROWS);
        int o = 0;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem)) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, kern, kW4a8Threads, smem) !=
                cudaSuccess)
            return 0;
        occ = o;
        device = ctx.device;
    }
    return occ;
}

// Fraction of the CTA slots of the GPU that the launch's waves keep busy.
inline double w4a8_wave_fill(int units, int per_sm, int sms) {
    if (per_sm < 1) return 0.0;
    const long long slots = static_cast<long long>(per_sm) * sms;
    const long long waves = (units + slots - 1) / slots;
    return static_cast<double>(units) / static_cast<double>(waves * slots);
}

template <int MT, int DT>
int launch_w4a8_dt(const DeviceCtx& ctx, const int8_t* A_i8, const float* s_a,
                   const void* packed, int M, int N, int K, void* Y, cudaStream_t stream) {
    // 16-channel CTAs (twice as many, each with twice the K slots) unless 32-channel
    // CTAs already fill every CTA slot of the GPU at least once; then whichever fills
    // the last wave better (32 on a tie: fewer K slots to reduce).
    const int units32 = w4a8_tiles(N), units16 = 2 * w4a8_tiles(N);
    const int occ32 = w4a8_occupancy<MT, DT, 32>(ctx), occ16 = w4a8_occupancy<MT, DT, 16>(ctx);
    if (occ32 < 1 || occ16 < 1) return -3;
    const double f32 = units32 >= occ32 * ctx.num_sms
                           ? w4a8_wave_fill(units32, occ32, ctx.num_sms) : 0.0;
    const double f16 = w4a8_wave_fill(units16, occ16, ctx.num_sms);
    if (f32 >= f16)
        return launch_w4a8_instance<MT, DT, 32>(ctx, A_i8, s_a, packed, M, N, K, Y, stream);
    return launch_w4a8_instance<MT, DT, 16>(ctx, A_i8, s_a, packed, M, N, K, Y, stream);
}

template <int MT>
int launch_w4a8_mt(const DeviceCtx& ctx, const int8_t* A_i8, const float* s_a,
                   const void* packed, int M, int N, int K, int dtype, void* Y,
                   cudaStream_t stream) {
    return dtype == 0 ? launch_w4a8_dt<MT, 0>(ctx, A_i8, s_a, packed, M, N, K, Y, stream)
                      : launch_w4a8_dt<MT, 1>(ctx, A_i8, s_a, packed, M, N, K, Y, stream);
}

}  // namespace

size_t w4a8_blob_bytes(int N, int K) {
    return static_cast<size_t>(w4a8_sw_offset(N, K)) + 4ull * w4a8_tiles(N) * kW4a8TileN;
}

int launch_w4a8_repack(const DeviceCtx& ctx, const uint32_t* qweight, const uint8_t* s_u8,
                       const uint8_t* off, const float* s_w, int N, int K, void* packed,
                       cudaStream_t stream) {
    const unsigned blocks = static_cast<unsigned>(w4a8_tiles(N) * (K / kW4a8Group));
    w4a8_repack_kernel<<<blocks, 128, 0, stream>>>(qweight, s_u8, off, s_w, N, K,
                                                    static_cast<uint8_t*>(packed), ctx.status);
    if (cudaGetLastError() != cudaSuccess) return -3;
    w4a8_fence_kernel<<<1, 32, 0, stream>>>();
    return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

int launch_w4a8_dequant_debug(const DeviceCtx& ctx, const void* packed, int N, int K,
                              void* W_out, cudaStream_t stream) {
    const unsigned blocks = static_cast<unsigned>(w4a8_tiles(N) * (K / kW4a8Group));
    w4a8_dequant_debug_kernel<<<blocks, 128, 0, stream>>>(
        static_cast<const uint8_t*>(packed), N, K, static_cast<int8_t*>(W_out), ctx.status);
    return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

int launch_w4a8_quantize(const DeviceCtx& ctx, const void* A, int M, int K, int dtype,
                         int8_t* A_i8, float* s_a, cudaStream_t stream) {
    (void)ctx;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(M), 1, 1);
    cfg.blockDim = dim3(kQuantThreads, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const uint16_t* a = static_cast<const uint16_t*>(A);
    const cudaError_t e =
        dtype == 0 ? cudaLaunchKernelEx(&cfg, w4a8_quantize_kernel<0>, a, K, A_i8, s_a)
                   : cudaLaunchKernelEx(&cfg, w4a8_quantize_kernel<1>, a, K, A_i8, s_a);
    return e == cudaSuccess ? 0 : -3;
}

int launch_w4a8_gemm(const DeviceCtx& ctx, const int8_t* A_i8, const float* s_a,
                     const void* packed, int M, int N, int K, int dtype, void* Y,
                     cudaStream_t stream) {
    if (M <= 1) return launch_w4a8_mt<1>(ctx, A_i8, s_a, packed, M, N, K, dtype, Y, stream);
    if (M <= 2) return launch_w4a8_mt<2>(ctx, A_i8, s_a, packed, M, N, K, dtype, Y, stream);
    if (M <= 4) return launch_w4a8_mt<4>(ctx, A_i8, s_a, packed, M, N, K, dtype, Y, stream);
    if (M <= 8) return launch_w4a8_mt<8>(ctx, A_i8, s_a, packed, M, N, K, dtype, Y, stream);
    if (M <= 16) return launch_w4a8_mt<16>(ctx, A_i8, s_a, packed, M, N, K, dtype, Y, stream);
    return -2;
}

}  // namespace w4g
