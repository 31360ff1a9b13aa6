// The fused W4A16 GEMM on the 5th-generation tensor cores (tcgen05), swap-AB form.
//
// One CTA computes a 128-channel x BM-row tile of Y^T = W . A^T over a K slice:
//
//   HBM --TMA bulk copy--> SMEM weight ring stage: packed 128x128 block(s)
//        (weights stream once, evict-first; "量化开销对比" §6.5; "W4A16 GEMM 算子浅析"
//         §"计算流水线的核心哲学", the HBM -> SMEM step)
//   L2/HBM --TMA tensor copy--> SMEM A ring stage: A tile (128-byte swizzle)
//   SMEM --dequant warps: LOP3 magic-bias unpack, sub/mul per pair--> TMEM (A operand)
//        ("W4A16 GEMM 算子浅析" §"寄存器解包黑魔法"; the group scale is applied here, on the
//         weight operand, as "量化开销对比" §6.2 requires)
//   tcgen05.mma.kind::f16 D[128 x BM] (fp32, TMEM) += W_tile[128 x 16] (TMEM) . A[BM x 16]^T
//        (the FP16 x FP16 -> FP32 MMA of the pipeline diagram; weights are the 128-row M
//         operand so that a decode batch of 1..16 tokens only pads the narrow N side)
//   epilogue: tcgen05.ld -> (split-K: each CTA of the cluster owns a slice of the 128
//        channels; the others push their fp32 partials for it into its shared memory
//        with bulk DSMEM copies; the owner sums them in rank order) -> x per-channel
//        factor -> optional + bias, activation, + residual -> round to dtype -> Y
//        ("量化开销对比" §6.2 "最后：累加器 × s_x → +bias → 写出", §6.6, §6.7 folding)
//
// The weights and the A tiles travel in two rings with their own producers and barriers:
// a weight slot is free again as soon as the dequant warps have read it (the unpacked
// tile lives in TMEM from then on), an A slot once the MMAs that read it have completed.
// So the weight stream runs ahead of the MMAs by the TMEM W buffers plus the weight ring,
// and neither waits for the other's slots to come back.
//
// Warp roles: warp 0 = weight producer; warps 1..NMI = MMA issuers (two for decode tiles
// of <= 32 rows and for 64- and 128-row whole-block tiles, taking even / odd 128-K blocks
// into two accumulators; warp 1 also allocates TMEM); warp NMI + 1 = A producer (decode tiles
// stream both rings from warp 0); then the dequant warps, 4 per warpgroup
// (warp w may only touch TMEM lanes 32*(w%4)..+31, so each warpgroup covers all 128
// lanes), which also run the epilogue.  The producer and issuer warps run their loops
// with all 32 lanes and let lane 0 issue, and the warp index and TMEM base are broadcast
// from lane 0, so that control flow and operand arithmetic are warp-uniform (uniform
// registers, fewer instructions per block).  Whole-block tiles: warpgroup g unpacks whole
// blocks g, g + NWG, ...; shared-block tiles: every warpgroup unpacks its chunks of every
// block; both through unpack routines templated on the group layout.  Each mbarrier has a
// single waiting party that passes every one of its phases (tfull per issuer and W buffer,
// tempty per warpgroup and W buffer), because a parity wait only tells the current phase
// from the one before it.
//
// Programmatic dependent launch: the prologue (barriers, TMEM, descriptor prefetch and,
// unless disabled, the header check), the weight stream and the unpack into TMEM run
// while the previous kernel in the stream finishes; A is read and Y written only after
// griddepcontrol.wait.  Every mbarrier wait is bounded; on expiry the CTA records a
// timeout, drains what it issued and exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstddef>
#include <cstring>
#include <mutex>

#include "dequant.cuh"
#include "epilogue.cuh"
#include "format.cuh"
#include "launch.h"
#include "ptx.cuh"

namespace w4g {

namespace {

constexpr int kCtrlBytes = 1024;

#ifndef W4A16_SMALL_TILE_WG
#define W4A16_SMALL_TILE_WG 2  // dequant warpgroups for 16- and 32-row tiles
#endif

constexpr int kFlagPrefetchW = 1;   // read header + first stages before the dependency wait

struct TcArgs {
    const uint8_t* packed;
    void* Y;
    int* status;
    int M, N, K, group;
    int kblocks;          // K / 128
    int splits;           // K slices = cluster size along x
    int a_stages;         // depth of the A ring
    int w_stages;         // depth of the weight ring
    int a_rows;           // rows per A chunk in shared memory (8, 16 or BM)
    int kps;              // 128-K blocks per stage of either ring (1 or 2)
    int a_2d;             // A loaded as one 2-D box per 64-K chunk (K not a multiple of 64)
    int slice_rows;       // channels owned per cluster rank (tc_slice_rows)
    int flags;
    uint32_t a_stage_bytes;
    uint32_t w_stage_bytes;
    uint32_t w_off;       // offset of the weight ring from the shared base (the A ring is at 0)
    uint32_t recv_off;    // offset of the split-K receive area from the shared base
    uint64_t timeout_ns;
    EpilogueArgs epi;     // bias / activation / residual applied to the fp32 result
};

template <int BM, bool kIL, int NWG>
struct TcShape {
    // MMA-issuing threads (one per warp).  A 128-row K=16 tcgen05.mma costs its issuing
    // thread tens of cycles, so narrow decode tiles (N = 16 or 32) and the 64- and
    // 128-row whole-block tiles split the blocks over two issuers, even blocks into
    // accumulator 0, odd into 1 (one issuer kept the tensor pipe of a 128-row tile ~70 %
    // busy).
    static constexpr int kNMI = (BM <= 32 || (kIL && (BM == 64 || BM == 128))) ? 2 : 1;
    static constexpr int kKps = BM <= 32 ? 2 : 1;          // 128-K blocks per ring stage
    // Decode tiles stream both rings from warp 0 (their A tiles are small and their K
    // slices short; an extra warp cost ~0.25 us per launch); larger tiles give the A ring
    // a producer warp of its own, so neither stream waits for the other's slots.
    static constexpr bool kOneProd = kKps == 2;
    static constexpr int kAProd = kOneProd ? 0 : 1 + kNMI;  // A producer warp
    static constexpr int kDq0 = (kOneProd ? 1 : 2) + kNMI;  // first dequant warp
    // kIL: each dequant warpgroup unpacks whole 128-K blocks (wg, wg + NWG, ...), so that
    // a block costs one warpgroup's per-block overhead (barrier waits, group constants)
    // and the groups' TMEM-store drains overlap; each group then owns a subset of the
    // weight ring's slots.  Otherwise every warpgroup takes its chunks of every block.
    static constexpr bool kInterleave = kIL;
    // warps that read each weight stage (and arrive on its empty barrier): one warpgroup
    // per block with whole-block groups, every warpgroup otherwise
    static constexpr int kWReaders(int nwg) { return (kIL ? 4 : 4 * nwg) * kKps; }
    static constexpr int kACol0 = kNMI * BM < 64 ? 64 : kNMI * BM;  // first W staging column
    // A stages an issuer advances per block it issues (two issuers with one block per
    // stage take every other stage)
    static constexpr int kSSteps = kNMI / kKps;
    // TMEM W buffers: as many as the CTA's TMEM share holds (256 columns when two CTAs
    // share an SM: tiles of up to 128 rows with two warpgroups; 512 for a CTA alone on an
    // SM: four warpgroups, or 256-row tiles), at most the control block's tfull slots
    static constexpr bool kShared = BM <= 128 && NWG <= 2;
    static constexpr int kTBufFit = (kShared ? 256 - kACol0 : 512 - kACol0) / 64;
    static constexpr int kTBuf = kTBufFit < 8 / kNMI ? kTBufFit : 8 / kNMI;
    static constexpr int kColsUsed = kACol0 + kTBuf * 64;
    static constexpr int kTmemCols = kColsUsed <= 32 ? 32 : kColsUsed <= 64 ? 64
                                   : kColsUsed <= 128 ? 128 : kColsUsed <= 256 ? 256 : 512;
};

template <int DT>
__device__ __forceinline__ uint16_t f32_to_dtype(float v) {
    if constexpr (DT == 0) return __half_as_ushort(__float2half_rn(v));
    else return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Unpack modes of a decode-tile block.
constexpr int kUnpackMagic = 0;     // exponent injection, pairs (k_2i, k_2i+1) shifted down
constexpr int kUnpackMagicX16 = 1;  // fp16: odd pairs masked in place (s/16 exact)
constexpr int kUnpackLut = 2;       // nibble -> value through a 16-entry shared table

// Chunks kC0, kC0 + kStep, ... (< 4) of one 128 x 128 block, one weight row r per thread;
// 32-K chunk c lands in TMEM columns taddr + 16 c.  kGS = 32-K chunks per quantisation
// group (4, 2, 1 for groups of 128, 64, 32).  lut: the shared 16-entry table (value bits
// of q = 0..15) used by kUnpackLut.
template <int DT, int kGS, int kMode, int kC0 = 0, int kStep = 1>
__device__ __forceinline__ void unpack_block_rows(const uint8_t* wb, int r,
                                                  const uint32_t (&sb)[4 / kGS],
                                                  const uint32_t (&zb)[4 / kGS], uint32_t taddr,
                                                  const uint16_t* lut) {
    uint32_t zp = 0, sp = 0, zp16 = 0, sp16 = 0;
#pragma unroll
    for (int c = kC0; c < 4; c += kStep) {
        if (c == kC0 || c / kGS != (c - kStep) / kGS) {  // a new group: its row constants
            const uint32_t z = (zb[c / kGS] >> ((r & 1) * 4)) & 0xFu;  // 8 when no zeros
            zp = kMode == kUnpackLut ? lut_zero_pair(lut, z) : zero_pair<DT>(z);
            sp = scale_pair(sb[c / kGS]);
            if constexpr (kMode == kUnpackMagicX16) {
                zp16 = zero_pair_x16(z);
                sp16 = scale_pair_div16(sp);
            }
        }
        const uint4 v = *reinterpret_cast<const uint4*>(wb + c * 2048 + r * 16);
        uint32_t out[16];
        if constexpr (kMode == kUnpackLut) {
            dequant_word_lut<DT>(v.x, lut, zp, sp, out + 0);
            dequant_word_lut<DT>(v.y, lut, zp, sp, out + 4);
            dequant_word_lut<DT>(v.z, lut, zp, sp, out + 8);
            dequant_word_lut<DT>(v.w, lut, zp, sp, out + 12);
        } else if constexpr (kMode == kUnpackMagicX16) {
            dequant_word_f16_x16(v.x, zp, sp, zp16, sp16, out + 0);
            dequant_word_f16_x16(v.y, zp, sp, zp16, sp16, out + 4);
            dequant_word_f16_x16(v.z, zp, sp, zp16, sp16, out + 8);
            dequant_word_f16_x16(v.w, zp, sp, zp16, sp16, out + 12);
        } else {
            dequant_word<DT>(v.x, zp, sp, out + 0);
            dequant_word<DT>(v.y, zp, sp, out + 4);
            dequant_word<DT>(v.z, zp, sp, out + 8);
            dequant_word<DT>(v.w, zp, sp, out + 12);
        }
        tmem_st16(taddr + c * 16, out);
    }
}

// Integer-operand unpack of one block (groups of 128: one scale and zero per block and
// row): the exact integers q - z go to TMEM; returns the row's scale, which the caller
// applies to the block's fp32 partial sum after the MMA.
template <int DT>
__device__ __forceinline__ float unpack_block_int(const uint8_t* wb, int r, uint32_t zoff,
                                                  bool has_z, uint32_t taddr) {
    const uint32_t z = has_z ? (wb[zoff + (r >> 1)] >> ((r & 1) * 4)) & 0xFu : 8u;
    const uint32_t zp = zero_pair<DT>(z);
    const uint32_t nz64 = DT == 0 ? neg64_pair(z) : 0u;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const uint4 v = *reinterpret_cast<const uint4*>(wb + c * 2048 + r * 16);
        uint32_t out[16];
        int_word<DT>(v.x, zp, nz64, out + 0);
        int_word<DT>(v.y, zp, nz64, out + 4);
        int_word<DT>(v.z, zp, nz64, out + 8);
        int_word<DT>(v.w, zp, nz64, out + 12);
        tmem_st16(taddr + c * 16, out);
    }
    return dtype_to_f32<DT>(reinterpret_cast<const uint16_t*>(wb + kNibbleBytes)[r]);
}

// Dequant modes of the tensor-core kernel (the alternatives for decode tiles only).
constexpr int kDqMagic = 0;  // exponent injection, one RNE of (q - z) s per weight
constexpr int kDqLut = 1;    // the 16-entry table, then the group's zero and scale
constexpr int kDqInt = 2;    // exact q - z to the MMA, the group scale on the fp32 partial

// Loads the block's group scales and zeros for row r, takes the fp16 x16 decision once for
// the whole block (warp vote), and unpacks it (kLut: through the shared table instead).
template <int DT, int kGS, bool kLut>
__device__ __forceinline__ void unpack_block(const uint8_t* wb, int r, uint32_t zoff,
                                             bool has_z, uint32_t taddr, const uint16_t* lut) {
    constexpr int kG = 4 / kGS;
    uint32_t sb[kG], zb[kG];
#pragma unroll
    for (int g = 0; g < kG; ++g) {
        sb[g] = reinterpret_cast<const uint16_t*>(wb + kNibbleBytes)[g * kTileN + r];
        zb[g] = has_z ? wb[zoff + g * (kTileN / 2) + (r >> 1)] : 0x88u;
    }
    if constexpr (kLut) {
        unpack_block_rows<DT, kGS, kUnpackLut>(wb, r, sb, zb, taddr, lut);
        return;
    }
    if constexpr (DT == 0) {
        bool exact = true;
#pragma unroll
        for (int g = 0; g < kG; ++g) {
            const uint32_t sp = scale_pair(sb[g]);
            exact = exact && f16_div16_exact(sp, scale_pair_div16(sp));
        }
        if (__all_sync(0xffffffffu, exact)) {
            unpack_block_rows<DT, kGS, kUnpackMagicX16>(wb, r, sb, zb, taddr, lut);
            return;
        }
    }
    unpack_block_rows<DT, kGS, kUnpackMagic>(wb, r, sb, zb, taddr, lut);
}

// Chunks kC0, kC0 + kStep, ... of a block, for tiles whose warpgroups share every block.
template <int DT, int kGS, int kC0, int kStep>
__device__ __forceinline__ void unpack_part(const uint8_t* wb, int r, uint32_t zoff,
                                            bool has_z, uint32_t taddr) {
    constexpr int kG = 4 / kGS;
    uint32_t sb[kG], zb[kG];
#pragma unroll
    for (int g = 0; g < kG; ++g) {
        sb[g] = reinterpret_cast<const uint16_t*>(wb + kNibbleBytes)[g * kTileN + r];
        zb[g] = has_z ? wb[zoff + g * (kTileN / 2) + (r >> 1)] : 0x88u;
    }
    if constexpr (DT == 0) {
        bool exact = true;
#pragma unroll
        for (int g = 0; g < kG; ++g) {
            const uint32_t sp = scale_pair(sb[g]);
            exact = exact && f16_div16_exact(sp, scale_pair_div16(sp));
        }
        if (__all_sync(0xffffffffu, exact)) {
            unpack_block_rows<DT, kGS, kUnpackMagicX16, kC0, kStep>(wb, r, sb, zb, taddr,
                                                                   nullptr);
            return;
        }
    }
    unpack_block_rows<DT, kGS, kUnpackMagic, kC0, kStep>(wb, r, sb, zb, taddr, nullptr);
}

// Warpgroup wg's chunks (wg, wg + NWG, ...) of a block, group layout resolved at compile time.
template <int DT, int NWG>
__device__ __forceinline__ void unpack_part_of(int wg, int gshift, const uint8_t* wb, int r,
                                               uint32_t zoff, bool has_z, uint32_t taddr) {
#define W4G_PART(C0)                                                                       \
    if (wg == C0) {                                                                        \
        if (gshift == 2) unpack_part<DT, 4, C0, NWG>(wb, r, zoff, has_z, taddr);           \
        else if (gshift == 1) unpack_part<DT, 2, C0, NWG>(wb, r, zoff, has_z, taddr);      \
        else unpack_part<DT, 1, C0, NWG>(wb, r, zoff, has_z, taddr);                       \
        return;                                                                            \
    }
    static_assert(NWG >= 1 && NWG <= 4, "one to four warpgroups");
    W4G_PART(0)
    if constexpr (NWG > 1) { W4G_PART(1) }
    if constexpr (NWG > 2) { W4G_PART(2) }
    if constexpr (NWG > 3) { W4G_PART(3) }
#undef W4G_PART
}

// kDq (the alternatives for decode tiles only): kDqLut unpacks through a 16-entry shared
// table of the values 0..15 instead of exponent injection (same results); kDqInt feeds
// the MMA the exact integers q - z and scales each block's fp32 partial (16-row tiles,
// groups of 128; the weights are not rounded to the activation dtype).
// kNoPushProbe: a failure-path check only (w4a16_debug_splitk_timeout_probe): cluster rank
// 0 pushes none of its partials, so the other ranks' bounded waits for them run out.
template <int BM, int NWG, int DT, int kDq = kDqMagic, bool kIL = (BM <= 32),
          bool kNoPushProbe = false>
__global__ void __launch_bounds__(32 * TcShape<BM, kIL, NWG>::kDq0 + 128 * NWG,
                                  (BM <= 64 && NWG <= 2) ? 2 : 1)
w4a16_tc_kernel(const __grid_constant__ CUtensorMap tmap_a, const TcArgs args) {
    using S = TcShape<BM, kIL, NWG>;
    constexpr int kTBuf = S::kTBuf;
    constexpr uint32_t kEpiThreads = 128 * NWG;
    constexpr int kNMI = S::kNMI;
    static_assert(S::kACol0 >= kNMI * BM, "accumulators overlap the W staging columns");
    static_assert(kNMI * kTBuf <= 8 && NWG * kTBuf <= 24, "control block barrier slots");
    static_assert(!S::kInterleave || NWG % S::kKps == 0, "whole-block groups: NWG % blocks per stage");
    constexpr bool kLut = kDq == kDqLut;
    constexpr bool kInt = kDq == kDqInt;
    static_assert(kDq == kDqMagic || S::kInterleave, "the alternatives exist for decode tiles");
    static_assert(!kInt || (BM == 16 && kNMI == 2 && NWG == 2), "integer operand: 16-row tiles");
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* base_ptr = smem_raw + (base - raw);
    // shared layout: [A ring][weight ring][split-K receive area][control block]
    const uint32_t ctrl_off = args.recv_off +
        (args.splits > 1 ? static_cast<uint32_t>((args.splits - 1) * BM * args.slice_rows * 4)
                         : 0u);
    const uint32_t ctrl = base + ctrl_off;
    uint8_t* ctrl_ptr = base_ptr + ctrl_off;
    const uint32_t wbase = base + args.w_off;
    // control block: wfull[16] (a weight stage landed) at 0, wempty[16] (a weight stage
    // read) at 128, tfull[issuer][W buffer] (8) at 256, aempty[16] (the MMAs that read an
    // A stage completed) at 320, accum / recv barriers and scalars at 448, kInt's dfull at
    // 496, tempty[warpgroup][W buffer] (24) at 528, afull[16] (an A stage landed) at 768
    const uint32_t wfull0 = ctrl, wempty0 = ctrl + 128, tfull0 = ctrl + 256;
    const uint32_t aempty0 = ctrl + 320, tempty0 = ctrl + 528, afull0 = ctrl + 768;
    uint16_t* lut = reinterpret_cast<uint16_t*>(ctrl_ptr + 960);  // 16 entries (kLut)
    // kInt: dfull[issuer][slot], the block's fp32 partial in D slot (issuer, slot) is done
    const uint32_t dfull0 = ctrl + 496;
    const uint32_t accum_bar = ctrl + 448;
    const uint32_t recv_bar = ctrl + 456;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ctrl_ptr + 464);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(ctrl_ptr + 468);
    int* info = reinterpret_cast<int*>(ctrl_ptr + 472);  // [0] flags or -1, [1] block bytes
    const float** cs_slot = reinterpret_cast<const float**>(ctrl_ptr + 480);

    // warp-uniform by construction (broadcast from lane 0), so values derived from it can
    // live in uniform registers (MMA and TMEM operands)
    const int warp = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x >> 5), 0);
    const int lane = static_cast<int>(threadIdx.x & 31);
    const int split = static_cast<int>(blockIdx.x);
    const int n_tile = static_cast<int>(blockIdx.y);
    const int m_tile = static_cast<int>(blockIdx.z);
    const int kb_per = args.kblocks / args.splits, kb_rem = args.kblocks % args.splits;
    const int kb0 = split * kb_per + (split < kb_rem ? split : kb_rem);
    const int nkb = kb_per + (split < kb_rem ? 1 : 0);
    const bool prefetch_w = (args.flags & kFlagPrefetchW) != 0;
    const uint32_t slice_bytes = static_cast<uint32_t>(BM * args.slice_rows * 4);

    // Thread 0 issues the header load first (its latency overlaps the barrier setup; with
    // weight prefetch disabled it must wait for the previous kernel instead), and warp 0
    // spreads the barrier initialisation over its lanes.
    uint4 hv[4];
    if (threadIdx.x == 0 && prefetch_w) {
        const uint4* hp = reinterpret_cast<const uint4*>(args.packed);
        for (int i = 0; i < 4; ++i) hv[i] = hp[i];
    }
    if (warp == 0) {
        if (lane == 0) {
            *abort_flag = 0;
        }
        for (int s = lane; s < args.w_stages; s += 32) {
            mbar_init(wfull0 + 8 * s, 1);
            mbar_init(wempty0 + 8 * s, S::kWReaders(NWG));  // one arrival per reading warp
        }
        for (int s = lane; s < args.a_stages; s += 32) {
            mbar_init(afull0 + 8 * s, 1);
            // an A stage is free once every issuer that read it has committed
            mbar_init(aempty0 + 8 * s, (kNMI == 2 && args.kps == 2) ? 2 : 1);
        }
        for (int t = lane; t < kNMI * kTBuf; t += 32)  // the warps that write a block's W tile
            mbar_init(tfull0 + 8 * t, S::kInterleave ? 4 : 4 * NWG);
        for (int t = lane; t < NWG * kTBuf; t += 32)
            mbar_init(tempty0 + 8 * t, 1);  // one MMA commit
        if (lane == 0) {
            mbar_init(accum_bar, kNMI);
            mbar_init(recv_bar, 1);
        }
        if (kInt && lane < 4) mbar_init(dfull0 + 8 * lane, 1);
        if (kLut && lane < 16) lut[lane] = value_bits<DT>(lane);
        fence_mbar_init();
        if (lane == 0) {
            if (args.splits > 1)  // partials of the other ranks for this rank's slice
                mbar_arrive_expect_tx(recv_bar, static_cast<uint32_t>(args.splits - 1) * slice_bytes);
            if (!prefetch_w) {
                grid_dep_wait();
                const uint4* hp = reinterpret_cast<const uint4*>(args.packed);
                for (int i = 0; i < 4; ++i) hv[i] = hp[i];
            }
            PackedHeader hl;  // the first 64 bytes: every field the check reads
            static_assert(offsetof(PackedHeader, total_bytes) + 8 <= 64, "header prefix");
            memcpy(&hl, hv, sizeof(hv));
            const int flags = check_header(&hl, args.N, args.K, args.group, DT);
            info[0] = flags;
            info[1] = flags < 0 ? 0 : static_cast<int>(hl.block_bytes);
            *cs_slot = (flags >= 0 && (flags & kFlagChannelScale))
                           ? reinterpret_cast<const float*>(args.packed + hl.cscale_offset)
                           : nullptr;
            if (flags < 0 && split == 0 && n_tile == 0 && m_tile == 0)
                record_status(args.status, kStatusFormat);
            prefetch_tensormap(&tmap_a);
        }
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(tmem_slot), S::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // peers may now target our barriers (their initialisation is fenced at cluster scope)
    if (args.splits > 1) cluster_arrive_relaxed();
    if (threadIdx.x == 0) grid_dep_launch();

    const uint32_t tmem = __shfl_sync(0xffffffffu, *tmem_slot, 0);
    const int flags = __shfl_sync(0xffffffffu, info[0], 0);
    const bool run = flags >= 0 && nkb > 0;
    const bool has_z = flags >= 0 && (flags & kFlagZeros) != 0;
    const uint32_t bb = static_cast<uint32_t>(__shfl_sync(0xffffffffu, info[1], 0));
    const float* cscale = *cs_slot;
    const uint64_t tlim = args.timeout_ns;
    const int kps = args.kps;
    const uint32_t a_chunk = static_cast<uint32_t>(args.a_rows) * 128u;   // one 64-K chunk of A
    const uint32_t a_bytes = 2u * static_cast<uint32_t>(kps) * a_chunk;  // A part of a stage
    const int nst = (nkb + kps - 1) / kps;                                // ring stages to stream

    // Drain after an abort: the last `depth` issued stages of a ring (every earlier one
    // was consumed, so it has landed) must land before the CTA may exit.
    auto drain = [&](uint32_t full_bars, int depth, int issued) {
        const int first = issued > depth ? issued - depth : 0;
        for (int i = first; i < issued; ++i) {
            int dummy = 0;
            (void)mbar_wait_bounded(full_bars + 8 * (i % depth),
                                    static_cast<uint32_t>(i / depth) & 1u, &dummy, nullptr, tlim);
        }
    };

    if (warp == 0 || warp == S::kAProd) {
        // ---------------- producers ----------------
        // Warp 0 streams the weight ring, warp kAProd the A ring (the same warp for decode
        // tiles).  The whole warp runs the loops (warp-uniform control and address
        // arithmetic); lane 0 arms the barriers and issues the copies.  Weight stage i =
        // blocks [i*kps, i*kps + nblk) as ONE bulk copy; A stage i = the 2*kps 64-K chunks
        // of A of those blocks as ONE 3-D box (or one 2-D box per chunk).  The packed
        // weights do not depend on the previous kernel (unless weight prefetch is off, in
        // which case the header was read after the dependency wait); A is written
        // upstream, so it is read only after the dependency wait.
        if (run) {
            const bool do_w = warp == 0, do_a = warp == S::kAProd;
            const uint64_t pol_w = policy_evict_first();
            const uint64_t pol_a = policy_evict_last();
            const uint8_t* wsrc = args.packed + kHeaderBytes +
                                  (static_cast<size_t>(n_tile) * args.kblocks + kb0) * bb;
            const int m0 = m_tile * BM;
            bool ok = true;
            // lane 0: the copies of weight / A stage i into ring slot `slot`
            auto copy_w = [&](int i, int slot) {
                const uint32_t fb = wfull0 + 8 * slot;
                const int left = nkb - i * kps;
                const uint32_t bytes = static_cast<uint32_t>(left < kps ? left : kps) * bb;
                mbar_arrive_expect_tx(fb, bytes);
                tma_bulk_g2s(wbase + static_cast<uint32_t>(slot) * args.w_stage_bytes,
                             wsrc + static_cast<size_t>(i) * kps * bb, bytes, fb, pol_w);
            };
            auto copy_a = [&](int i, int slot) {
                const uint32_t st = base + static_cast<uint32_t>(slot) * args.a_stage_bytes;
                const uint32_t ab = afull0 + 8 * slot;
                const int kchunk = (kb0 + i * kps) * 2;  // first 64-K chunk of the stage
                mbar_arrive_expect_tx(ab, a_bytes);
                if (args.a_2d) {  // chunk q at st + q * a_chunk; the K tail zero-filled
                    for (int q = 0; q < 2 * kps; ++q)
                        tma_tensor_2d_g2s(st + static_cast<uint32_t>(q) * a_chunk, &tmap_a,
                                          (kchunk + q) * 64, m0, ab, pol_a);
                } else {
                    tma_tensor_3d_g2s(st, &tmap_a, 0, m0, kchunk, ab, pol_a);
                }
            };
            // warp-wide: wait for the slot (after its first use), then lane 0 copies
            int wi = 0, ws = 0;  // next weight stage, its slot and the parity of that use
            uint32_t wph = 0;
            auto issue_w = [&]() {
                if (wi >= args.w_stages)
                    ok = ok && mbar_wait_warp(wempty0 + 8 * ws, wph ^ 1u, abort_flag,
                                              args.status, tlim);
                if (!ok) return;
                if (lane == 0) copy_w(wi, ws);
                ++wi;
                if (++ws == args.w_stages) { ws = 0; wph ^= 1u; }
            };
            int ai = 0, as = 0;  // the same for the A ring
            uint32_t aph = 0;
            auto issue_a = [&]() {
                if (ai >= args.a_stages)
                    ok = ok && mbar_wait_warp(aempty0 + 8 * as, aph ^ 1u, abort_flag,
                                              args.status, tlim);
                if (!ok) return;
                if (lane == 0) copy_a(ai, as);
                ++ai;
                if (++as == args.a_stages) { as = 0; aph ^= 1u; }
            };
            // Lane 0 first issues the weight stages that need no slot back and, after the
            // dependency wait, the A stages that need none, in straight loops (0.1 us per
            // decode launch faster than issuing them warp-wide).  Then the warp always
            // takes the copy whose slot is released first: weight stage wi waits for the
            // unpack of stage wi - w_stages, A stage ai for the MMAs of stage ai -
            // a_stages; a stage's unpack precedes its MMAs, so the lower stage index (the
            // weight stage on a tie) goes first.  With one warp for both rings every wait
            // is then for a stage whose own copies were issued earlier: no wait can block
            // a copy that it depends on.
            const int nw = do_w ? nst : 0, na = do_a ? nst : 0;  // stages this warp streams
            const int pw = nw < args.w_stages ? nw : args.w_stages;
            const int pa = na < args.a_stages ? na : args.a_stages;
            if (lane == 0)
                for (int i = 0; i < pw; ++i) copy_w(i, i);
            if (do_a) {
                grid_dep_wait();
                if (lane == 0)
                    for (int i = 0; i < pa; ++i) copy_a(i, i);
            }
            __syncwarp();
            wi = ws = pw;
            if (ws == args.w_stages) { ws = 0; wph = 1u; }
            ai = as = pa;
            if (as == args.a_stages) { as = 0; aph = 1u; }
            while (ok && (wi < nw || ai < na)) {
                if (wi < nw && (ai >= na || wi - args.w_stages <= ai - args.a_stages))
                    issue_w();
                else
                    issue_a();
            }
            if (lane == 0 && (!ok || *abort_flag)) {
                if (do_w) drain(wfull0, args.w_stages, wi);
                if (do_a) drain(afull0, args.a_stages, ai);
            }
        }
        __syncwarp();
        if (args.splits > 1) {  // phase 0 (peers' barriers ready), then arrive for the exit
            cluster_wait_acquire();
            cluster_arrive_relaxed();
        }
    } else if (warp <= kNMI) {
        // ---------------- MMA issuers (one thread per warp) ----------------
        const int k = warp - 1;  // issuer index: blocks k, k + kNMI, ...
        // The whole warp runs the loop (warp-uniform control and operand arithmetic);
        // lane 0 issues the MMAs and the commits that track them.
        if (run) {
            constexpr uint32_t idesc = idesc_f16(DT, 128, BM);
            // Descriptor of chunk c, 16-K step q of the A tile in a stage = descriptor of
            // the stage base + (c * a_chunk + 32 q) / 16; only the start address moves.
            const uint64_t chunk16 = a_chunk >> 4;
            const uint32_t dacc = tmem + static_cast<uint32_t>(k * BM);  // this issuer's D
            bool ok = true;
            // Two issuers and two blocks per stage: issuer k owns block b = k of every
            // stage.  Two issuers and one block per stage: issuer k takes stages k, k + 2,
            // ... (the host keeps the A ring depth even, so each A slot has one waiting
            // issuer).
            int s = (kNMI == 2 && S::kKps == 1) ? k : 0;
            int b = (kNMI == 2 && S::kKps == 2) ? k : 0, t = k;
            uint32_t ph = 0;
            uint32_t fpar = 0;  // bit t: parity of this issuer's next wait on tfull[k][t]
            for (int i = k; i < nkb; i += kNMI) {   // i: 128-K block
                // the A stage of block i (its weights are in TMEM once tfull completes)
                ok = (kNMI == 1 && b != 0) ||
                     mbar_wait_spin_warp(afull0 + 8 * s, ph, abort_flag, args.status, tlim);
                ok = ok && mbar_wait_spin_warp(tfull0 + 8 * (k * kTBuf + t), (fpar >> t) & 1u,
                                               abort_flag, args.status, tlim);
                fpar ^= 1u << t;
                if (!ok) break;
                tc_fence_after();
                const uint64_t d0 = sw128_desc(base + static_cast<uint32_t>(s) * args.a_stage_bytes) +
                                    static_cast<uint64_t>(2 * b) * chunk16;
                const uint64_t d1 = d0 + chunk16;
                const uint32_t a0 = tmem + S::kACol0 + t * 64;
                // the W buffer is free for its next block, i + kTBuf (unpacked by warpgroup
                // (i + kTBuf) % NWG when warpgroups take whole blocks, else by all)
                const uint32_t te =
                    tempty0 + 8 * ((S::kInterleave ? (i + kTBuf) % NWG : 0) * kTBuf + t);
                const bool stage_done = kNMI == 2 || b + 1 == kps || i == nkb - 1;
                // kInt: block i's own fp32 partial, in D slot (k, (i / kNMI) & 1)
                const uint32_t dslot = (k * 2 + ((i / kNMI) & 1)) * BM;
                const uint32_t dd = kInt ? tmem + dslot : dacc;
                if constexpr (kInt) {
                    if (lane == 0) {
                        tc_mma_ts(dd, a0, d0, idesc, 0u);
                        tc_mma_ts(dd, a0 + 8, d0 + 2, idesc, 1u);
                        tc_mma_ts(dd, a0 + 16, d0 + 4, idesc, 1u);
                        tc_mma_ts(dd, a0 + 24, d0 + 6, idesc, 1u);
                        tc_mma_ts(dd, a0 + 32, d1, idesc, 1u);
                        tc_mma_ts(dd, a0 + 40, d1 + 2, idesc, 1u);
                        tc_mma_ts(dd, a0 + 48, d1 + 4, idesc, 1u);
                        tc_mma_ts(dd, a0 + 56, d1 + 6, idesc, 1u);
                        tc_commit(te);
                        tc_commit(dfull0 + dslot / 2);  // 8 bytes per (k, slot)
                        if (stage_done) tc_commit(aempty0 + 8 * s);
                    }
                } else {  // the whole warp executes it, lane 0 issues and commits
                    const uint32_t av[8] = {a0, a0 + 8, a0 + 16, a0 + 24,
                                            a0 + 32, a0 + 40, a0 + 48, a0 + 56};
                    const uint64_t bv[8] = {d0, d0 + 2, d0 + 4, d0 + 6, d1, d1 + 2, d1 + 4, d1 + 6};
                    tc_mma_block_lane0(dd, av, bv, idesc, i >= kNMI ? 1u : 0u, te,
                                       stage_done ? aempty0 + 8 * s : 0u);
                }
                __syncwarp();
                t += kNMI;
                if (t >= kTBuf) t -= kTBuf;
                if (kNMI == 1) b = stage_done ? 0 : b + 1;
                if (stage_done) {
                    s += S::kSSteps;
                    if (s >= args.a_stages) { s -= args.a_stages; ph ^= 1u; }
                }
            }
            if (lane == 0) {
                tc_commit(accum_bar);
            }
            if (!ok && lane == 0) {  // no MMA may still read TMEM/SMEM when the CTA exits
                int dummy = 0;
                (void)mbar_wait_bounded(accum_bar, 0, &dummy, nullptr, tlim);
            }
        } else if (lane == 0) {
            tc_commit(accum_bar);  // no MMAs to track: arrive at once
        }
        __syncwarp();
        if (args.splits > 1) {
            cluster_wait_acquire();
            cluster_arrive_relaxed();
        }
    } else {
        // ---------------- dequant warps ----------------
        const int q = warp & 3;                 // TMEM lane quarter of this warp
        const int wg = (warp - S::kDq0) >> 2;   // dequant warpgroup
        const int r = q * 32 + lane;            // weight row of the tile == TMEM lane
        const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
        const uint32_t zoff = kNibbleBytes + scale_bytes(args.group);
        bool ok = run;
        const int gshift = args.group == 128 ? 2 : (args.group == 64 ? 1 : 0);  // chunk -> group
        // Decode tiles: warpgroup wg unpacks whole 128-K blocks wg, wg + NWG, ..., so one
        // group's TMEM stores drain while another unpacks.  Larger tiles: every warpgroup
        // unpacks chunks wg, wg + NWG, ... of every block.  A parity wait is only
        // meaningful for the current or the immediately preceding phase of an mbarrier,
        // so every barrier has a single waiting party that takes part in each of its
        // phases: issuer k waits on tfull[k][t] (its own blocks in W buffer t), warpgroup
        // w on tempty[w][t] (the MMA of the block before its own next use of buffer t;
        // one shared party when all groups unpack every block), and each warpgroup passes
        // every phase of the weight ring slots it reads (the host keeps the weight ring
        // depth a multiple of NWG / blocks-per-stage when groups take whole blocks).
        constexpr int kBStep = S::kInterleave ? NWG : 1;         // block stride of a group
        // With whole blocks per group and kKps blocks per ring stage, warpgroup wg reads
        // block wg % kKps of weight stages wg / kKps, wg / kKps + NWG / kKps, ... (the host
        // keeps the weight ring depth a multiple of NWG / kKps) and uses W buffers wg,
        // wg + NWG, ... mod kTBuf.
        constexpr int kSStep = S::kInterleave ? NWG / S::kKps : 1;  // ring slots per block step
        const int tw = S::kInterleave ? wg : 0;                  // tempty party
        int s = S::kInterleave ? wg / S::kKps : 0;  // weight slot of block i, and the parity
        uint32_t ph = 0;                            // of that use of the slot
        int b = S::kInterleave ? wg % S::kKps : 0;  // block i's place in its stage
        int t = S::kInterleave ? wg % kTBuf : 0;    // its W buffer
        uint32_t epar = 0;      // bit t: parity of this warp's next wait on tempty[tw][t]
        // kInt: this thread's running sum over its group's blocks (row r, BM columns), the
        // scale of the block unpacked last, and that block's place in the group's order
        float iacc[kInt ? BM : 1];
#pragma unroll
        for (int m = 0; m < (kInt ? BM : 1); ++m) iacc[m] = 0.0f;
        float s_last = 0.0f;
        int jn = 0;             // blocks this group has unpacked
        // adds block j's partial (D slot (wg, j & 1), ready when dfull's phase j / 2 is)
        auto rescale = [&](int j, float sc) {
            if constexpr (kInt) {
                const uint32_t sl = static_cast<uint32_t>(j & 1);
                ok = ok && mbar_wait_warp(dfull0 + 8 * (wg * 2 + sl), (j >> 1) & 1, abort_flag,
                                          args.status, tlim);
                if (!ok) return;
                tc_fence_after();
                uint32_t v[16];
                tmem_ld16(tmem + lane_base + (wg * 2 + sl) * BM, v);
                tmem_wait_ld();
#pragma unroll
                for (int m = 0; m < BM; ++m) iacc[m] = fmaf(__uint_as_float(v[m]), sc, iacc[m]);
            }
        };
        for (int i = S::kInterleave ? wg : 0; i < nkb && ok; i += kBStep) {   // 128-K block
            if (S::kInterleave || b == 0)  // (s, b, t) advance at the loop end
                ok = mbar_wait_warp(wfull0 + 8 * s, ph, abort_flag, args.status, tlim);
            if (ok && i >= kTBuf) {
                ok = mbar_wait_warp(tempty0 + 8 * (tw * kTBuf + t), (epar >> t) & 1u, abort_flag,
                                    args.status, tlim);
                epar ^= 1u << t;
            }
            if (!ok) break;
            const uint8_t* wb = base_ptr + args.w_off +
                                static_cast<size_t>(s) * args.w_stage_bytes +
                                static_cast<size_t>(b) * bb;
            float s_cur = 0.0f;  // kInt: the block's scale for row r
            if constexpr (S::kInterleave) {  // whole block by this warpgroup
                const uint32_t taddr = tmem + lane_base + S::kACol0 + t * 64;
                if constexpr (kInt) s_cur = unpack_block_int<DT>(wb, r, zoff, has_z, taddr);
                else if (gshift == 2) unpack_block<DT, 4, kLut>(wb, r, zoff, has_z, taddr, lut);
                else if (gshift == 1) unpack_block<DT, 2, kLut>(wb, r, zoff, has_z, taddr, lut);
                else unpack_block<DT, 1, kLut>(wb, r, zoff, has_z, taddr, lut);
            } else {  // this warpgroup's chunks of the block
                unpack_part_of<DT, NWG>(wg, gshift, wb, r, zoff, has_z,
                                        tmem + lane_base + S::kACol0 + t * 64);
            }
            // every lane's shared-memory reads of the block are done (their values are in
            // the TMEM stores): the weight slot may be refilled
            __syncwarp();
            if (lane == 0) mbar_arrive(wempty0 + 8 * s);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tfull0 + 8 * ((i % kNMI) * kTBuf + t));
            if constexpr (kInt) {  // the previous block's partial, while this one is in the MMA
                if (jn > 0) rescale(jn - 1, s_last);
                s_last = s_cur;
                ++jn;
            }
            if constexpr (S::kInterleave) {
                s += kSStep;
                if (s >= args.w_stages) { s -= args.w_stages; ph ^= 1u; }
                t += NWG % kTBuf;
                if (t >= kTBuf) t -= kTBuf;
            } else {
                if (++t == kTBuf) t = 0;
                if (++b == args.kps) {
                    b = 0;
                    if (++s == args.w_stages) { s = 0; ph ^= 1u; }
                }
            }
        }

        if (kInt && ok && jn > 0) rescale(jn - 1, s_last);

        // ---------------- epilogue ----------------
        const int R = args.slice_rows;
        float* part = reinterpret_cast<float*>(base_ptr);  // [slice][BM][R] when split
        ok = ok && mbar_wait_warp(accum_bar, 0, abort_flag, args.status, tlim);
        // kInt: each group's sum goes to TMEM where the epilogue expects the two issuers'
        // accumulators (columns d_base and d_base + BM, in the now idle W buffer area)
        uint32_t d_base = 0;
        if constexpr (kInt) {
            d_base = S::kACol0;
            if (ok) {
                tc_fence_after();
                uint32_t v[16];
#pragma unroll
                for (int m = 0; m < 16; ++m) v[m] = __float_as_uint(iacc[m]);
                tmem_st16(tmem + lane_base + d_base + wg * BM, v);
                tmem_wait_st();
            }
            tc_fence_before();
            named_bar_sync(2, kEpiThreads);  // both groups' sums are in place
        }
        if (ok) {
            tc_fence_after();
            const int n = n_tile * kTileN + r;
            uint16_t* Y = static_cast<uint16_t*>(args.Y);
            if (args.splits == 1) grid_dep_wait();  // Y may still be in use upstream
            const bool n_ok = n < args.N;  // rows past N are padding
            const float cs = (args.splits == 1 && cscale && n_ok) ? cscale[n] : 1.0f;
            const float bias_n = (args.splits == 1 && args.epi.bias && n_ok)
                                     ? dtype_to_f32<DT>(args.epi.bias[n]) : 0.0f;
            const int pslice = r / R, prow = r - pslice * R;
            // D columns e*16 .. e*16+15 of this thread's channel (both accumulators added)
            auto load_d = [&](int e, uint32_t (&v)[16]) {
                tmem_ld16(tmem + lane_base + d_base + e * 16, v);
                if (kNMI == 2 && nkb > 1) {  // add the odd-block accumulator
                    uint32_t v1[16];
                    tmem_ld16(tmem + lane_base + d_base + BM + e * 16, v1);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        v[j] = __float_as_uint(__uint_as_float(v[j]) + __uint_as_float(v1[j]));
                } else {
                    tmem_wait_ld();
                }
            };
            if (args.splits > 1) {
#pragma unroll 1
                for (int e = wg; e < BM / 16; e += NWG) {
                    uint32_t v[16];
                    load_d(e, v);
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        part[(pslice * BM + e * 16 + j) * R + prow] = __uint_as_float(v[j]);
                }
            } else if (BM >= 64 &&
                       ((reinterpret_cast<uintptr_t>(args.Y) |
                         reinterpret_cast<uintptr_t>(args.epi.residual)) & 15u) == 0) {
                // Larger tiles: each warp stages its 32 channels x 16 rows of A through
                // shared memory (the idle ring) and stores 8 channels per 16-byte access,
                // reading the residual the same way; the fp32 operations and their order
                // are those of the paths below, so the results are the same bits.
                const int act = args.epi.act;
                const uint16_t* rp = args.epi.residual;
                float* T = reinterpret_cast<float*>(base_ptr) + (warp - S::kDq0) * 512;  // [16][32]
                const int n0w = n_tile * kTileN + q * 32;  // first channel of this warp
                // The residual of the next 16-row group is loaded while this group is
                // computed and stored, so that its latency is not paid once per group.
                // Groups hold disjoint rows, and a thread reads an element of the residual
                // only before it writes that element of Y, so Y may be the residual itself.
                auto load_res8 = [&](int e, uint4 (&rv)[2]) {
#pragma unroll
                    for (int p = 0; p < 2; ++p) {
                        const int m = m_tile * BM + e * 16 + p * 8 + (lane >> 2);
                        const int nn = n0w + (lane & 3) * 8;
                        rv[p] = (m < args.M && nn < args.N)
                                    ? *reinterpret_cast<const uint4*>(
                                          rp + static_cast<size_t>(m) * args.N + nn)
                                    : make_uint4(0u, 0u, 0u, 0u);
                    }
                };
                uint4 rnext[2] = {make_uint4(0u, 0u, 0u, 0u), make_uint4(0u, 0u, 0u, 0u)};
                if (rp && wg < BM / 16) load_res8(wg, rnext);
#pragma unroll 1
                for (int e = wg; e < BM / 16; e += NWG) {
                    const uint4 rcur[2] = {rnext[0], rnext[1]};
                    if (rp && e + NWG < BM / 16) load_res8(e + NWG, rnext);
                    uint32_t v[16];
                    load_d(e, v);  // warp-collective: every lane, padded rows included
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const float y = __uint_as_float(v[j]) * cs + bias_n;
                        T[j * 32 + lane] = act == kActNone ? y : apply_activation(y, act);
                    }
                    __syncwarp();
#pragma unroll
                    for (int p = 0; p < 2; ++p) {
                        const int jm = p * 8 + (lane >> 2);  // row of A within the group
                        const int nb = (lane & 3) * 8;       // first of 8 channels
                        const int m = m_tile * BM + e * 16 + jm;
                        const int nn = n0w + nb;             // N % 8 == 0: 8 valid or none
                        if (m < args.M && nn < args.N) {
                            const float4 lo = *reinterpret_cast<const float4*>(T + jm * 32 + nb);
                            const float4 hi =
                                *reinterpret_cast<const float4*>(T + jm * 32 + nb + 4);
                            float f[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
                            const size_t o = static_cast<size_t>(m) * args.N + nn;
                            if (rp) {
                                const uint4 rv = rcur[p];
                                const uint32_t rw[4] = {rv.x, rv.y, rv.z, rv.w};
#pragma unroll
                                for (int h = 0; h < 8; ++h)
                                    f[h] += dtype_to_f32<DT>(
                                        static_cast<uint16_t>(rw[h >> 1] >> ((h & 1) * 16)));
                            }
                            uint32_t ow[4];
#pragma unroll
                            for (int h = 0; h < 4; ++h)
                                ow[h] = static_cast<uint32_t>(f32_to_dtype<DT>(f[2 * h])) |
                                        (static_cast<uint32_t>(f32_to_dtype<DT>(f[2 * h + 1])) << 16);
                            *reinterpret_cast<uint4*>(Y + o) = make_uint4(ow[0], ow[1], ow[2], ow[3]);
                        }
                    }
                    __syncwarp();  // the tile is read before the next group overwrites it
                }
            } else if (!args.epi.residual) {
                const int act = args.epi.act;
#pragma unroll 1
                for (int e = wg; e < BM / 16; e += NWG) {
                    uint32_t v[16];
                    load_d(e, v);  // warp-collective: every lane, padded rows included
                    if (!n_ok) continue;  // a padded row: nothing to store
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int m = m_tile * BM + e * 16 + j;
                        const float y = __uint_as_float(v[j]) * cs + bias_n;
                        if (m < args.M)
                            Y[static_cast<size_t>(m) * args.N + n] =
                                f32_to_dtype<DT>(act == kActNone ? y : apply_activation(y, act));
                    }
                }
            } else {
                // The residual may be Y itself, so its loads cannot move past earlier
                // stores: the next group's 16 values are read before this group is stored.
                const uint16_t* rp = args.epi.residual;
                auto load_res = [&](int e, float (&r)[16]) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int m = m_tile * BM + e * 16 + j;
                        r[j] = (m < args.M && n_ok)
                                   ? dtype_to_f32<DT>(rp[static_cast<size_t>(m) * args.N + n])
                                   : 0.0f;
                    }
                };
                float rnext[16];
                if (wg < BM / 16) load_res(wg, rnext);
#pragma unroll 1
                for (int e = wg; e < BM / 16; e += NWG) {
                    float res[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) res[j] = rnext[j];
                    if (e + NWG < BM / 16) load_res(e + NWG, rnext);
                    uint32_t v[16];
                    load_d(e, v);  // warp-collective: every lane, padded rows included
                    if (!n_ok) continue;
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int m = m_tile * BM + e * 16 + j;
                        if (m < args.M)
                            Y[static_cast<size_t>(m) * args.N + n] = f32_to_dtype<DT>(
                                apply_activation(__uint_as_float(v[j]) * cs + bias_n, args.epi.act) +
                                res[j]);
                    }
                }
            }
        }
        if (args.splits > 1) {
            // Push our partial of every other rank's slice into that rank's receive area.
            fence_proxy_async_smem();
            named_bar_sync(1, kEpiThreads);
            cluster_wait_acquire();  // every peer has initialised its receive barrier
            const uint32_t rank = cluster_ctarank();
            if (warp == S::kDq0) {  // lane p sends the slice of rank p
                const int p = lane;
                if (p < args.splits && p != static_cast<int>(rank) &&
                    !(kNoPushProbe && rank == 0)) {
                    const uint32_t src = base + static_cast<uint32_t>(p) * slice_bytes;
                    // rank's slot in p's receive area (one slot per other rank)
                    const uint32_t slot = rank < static_cast<uint32_t>(p) ? rank : rank - 1u;
                    const uint32_t dst =
                        map_to_rank(base + args.recv_off + slot * slice_bytes, p);
                    bulk_s2cluster(dst, src, slice_bytes, map_to_rank(recv_bar, p));
                    bulk_commit();
                    bulk_wait_read_all();
                }
                __syncwarp();
            }
            // Sum this rank's slice over all ranks, in rank order, and store it.  Every
            // peer pushes its partial even after a failure of its own (a peer is late by
            // at most one wait limit), so this wait is bounded by time only, twice the
            // limit, not by this CTA's abort flag: the pushes are allowed to land before
            // the CTA may leave.  Arriving at the exit phase of the cluster barrier right
            // after it tells the peers that their pushes into this CTA have landed, i.e.
            // that their sources have been read.
            volatile int no_abort = 0;
            const bool got = mbar_wait_warp(recv_bar, 0, &no_abort, args.status, 2 * tlim);
            cluster_arrive_relaxed();
            if (ok && got) {
                grid_dep_wait();
                // Thread t owns the 4 channels 4 (t % nq) .. + 3 of this rank's slice and
                // rows t / nq, t / nq + mstep, ...: 16-byte reads of the partials, 8-byte
                // stores of Y, the channel constants read once (R, r0 and N are multiples
                // of 4, so the quads are aligned and never straddle the slice's end).
                const int r0 = static_cast<int>(rank) * R;
                const int nr = min(min(kTileN, r0 + R), args.N - n_tile * kTileN) - r0;
                const int mvalid = min(BM, args.M - m_tile * BM);
                const float* recvp = reinterpret_cast<const float*>(base_ptr + args.recv_off);
                uint16_t* Y = static_cast<uint16_t*>(args.Y);
                const int tid = static_cast<int>(threadIdx.x) - 32 * S::kDq0;
                if constexpr (BM <= 32) {
                    // Decode tiles: at most 32 rows of a slice, one element per thread and
                    // pass.  (A compact loop: this tail runs once per CTA on the critical
                    // path, and the 4-channel form below measured 0.2 us slower here.)
                    for (int e = tid; nr > 0 && e < nr * mvalid;
                         e += static_cast<int>(kEpiThreads)) {
                        const int ml = e / nr;
                        const int j = e - ml * nr;
                        float acc = 0.0f;
                        for (int p = 0; p < args.splits; ++p) {
                            const int slot = p < static_cast<int>(rank) ? p : p - 1;
                            const float* src = p == static_cast<int>(rank)
                                                   ? part + (static_cast<int>(rank) * BM + ml) * R
                                                   : recvp + (slot * BM + ml) * R;
                            acc += src[j];
                        }
                        const int n = n_tile * kTileN + r0 + j;
                        if (cscale) acc *= cscale[n];
                        const float bias_n =
                            args.epi.bias ? dtype_to_f32<DT>(args.epi.bias[n]) : 0.0f;
                        const size_t o = static_cast<size_t>(m_tile * BM + ml) * args.N + n;
                        Y[o] = f32_to_dtype<DT>(apply_epilogue<DT>(acc, bias_n, args.epi, o));
                    }
                } else {
                const int nq = nr > 0 ? nr / 4 : 0;
                const int mstep = nq > 0 ? static_cast<int>(kEpiThreads) / nq : 0;
                const int tq = nq > 0 ? tid % nq : 0;
                const int mfirst = nq > 0 ? tid / nq : 0;
                if (nq > 0 && mfirst < mstep) {
                    const int j = 4 * tq;
                    const int n = n_tile * kTileN + r0 + j;
                    float csq[4], bq[4];
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        csq[h] = cscale ? cscale[n + h] : 1.0f;
                        bq[h] = args.epi.bias ? dtype_to_f32<DT>(args.epi.bias[n + h]) : 0.0f;
                    }
                    for (int ml = mfirst; ml < mvalid; ml += mstep) {
                        float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                        for (int p = 0; p < args.splits; ++p) {  // rank order
                            const int slot = p < static_cast<int>(rank) ? p : p - 1;
                            const float* src = p == static_cast<int>(rank)
                                                   ? part + (static_cast<int>(rank) * BM + ml) * R
                                                   : recvp + (slot * BM + ml) * R;
                            const float4 v = *reinterpret_cast<const float4*>(src + j);
                            acc[0] += v.x;
                            acc[1] += v.y;
                            acc[2] += v.z;
                            acc[3] += v.w;
                        }
                        const size_t o = static_cast<size_t>(m_tile * BM + ml) * args.N + n;
                        uint32_t w[2];
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const float y0 = apply_epilogue<DT>(acc[2 * h] * csq[2 * h],
                                                                bq[2 * h], args.epi, o + 2 * h);
                            const float y1 = apply_epilogue<DT>(acc[2 * h + 1] * csq[2 * h + 1],
                                                                bq[2 * h + 1], args.epi,
                                                                o + 2 * h + 1);
                            w[h] = static_cast<uint32_t>(f32_to_dtype<DT>(y0)) |
                                   (static_cast<uint32_t>(f32_to_dtype<DT>(y1)) << 16);
                        }
                        *reinterpret_cast<uint2*>(Y + o) = make_uint2(w[0], w[1]);
                    }
                }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    // A cluster rank must not exit while a peer may still push partials into its shared
    // memory, or read its own partials out of it: every rank arrives at the exit phase
    // once the pushes into it have landed (or the bounded wait for them ran out), and
    // leaves only when all ranks have arrived.  In the normal case the peers arrived
    // long before this rank's own stores are done, so the wait costs nothing.
    if (args.splits > 1) {
        cluster_wait_acquire();
        // Every peer has now issued its push into this CTA; if the receive wait above
        // ran out, give those pushes (bounded) time to land before the CTA exits.
        if (threadIdx.x == 0) {
            int dummy = 0;
            (void)mbar_wait_bounded(recv_bar, 0, &dummy, nullptr, tlim);
        }
    }
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

template <int BM, int NWG, int DT, int DQ = kDqMagic, bool IL = (BM <= 32), bool PROBE = false>
int launch_tc_instance(const DeviceCtx& ctx, const void* A, const void* packed, int M, int N,
                       int K, int group, void* Y, const GemmPlan& plan,
                       const EpilogueArgs& epi, cudaStream_t stream,
                       uint64_t timeout_ns = 0) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return -3;
    const int a_rows = tc_a_rows(BM, M);
    const int kps = tc_blocks_per_stage(BM);
    // A viewed as [K/64][M][64]: one box = 2*kps chunks of 64 K x a_rows rows, landing in
    // shared memory chunk-major, each chunk a run of 128-byte-swizzled 8-row atoms.  A
    // chunk past K is outside the view and arrives as zeros.  If K is not a multiple of
    // 64 that view does not exist: A is then the plain 2-D [M][K] tensor and every 64-K
    // chunk is its own box (the part past K zero-filled), in the same shared layout.
    const bool a_2d = K % 64 != 0;
    // Encoding a tensor map costs host time on every call; the encoded map depends only
    // on the values below, so each host thread keeps the last few it made.
    struct MapEntry {
        CUtensorMap map;
        const void* ptr;
        int M, K, a_rows, kps, dt, valid;
    };
    thread_local MapEntry cache[8];
    thread_local int cache_next = 0;
    const CUtensorMap* mp = nullptr;
    for (const MapEntry& e : cache)
        if (e.valid && e.ptr == A && e.M == M && e.K == K && e.a_rows == a_rows && e.kps == kps &&
            e.dt == DT) {
            mp = &e.map;
            break;
        }
    if (!mp) {
        MapEntry& e = cache[cache_next];
        cache_next = (cache_next + 1) % 8;
        e.valid = 0;
        const auto dt = DT == 0 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
        CUresult cr;
        if (!a_2d) {
            const cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(M), static_cast<cuuint64_t>(K / 64)};
            const cuuint64_t strides[2] = {static_cast<cuuint64_t>(K) * 2, 128};
            const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(a_rows),
                                       static_cast<cuuint32_t>(2 * kps)};
            const cuuint32_t estr[3] = {1, 1, 1};
            cr = enc(&e.map, dt, 3, const_cast<void*>(A), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        } else {
            const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M)};
            const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
            const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(a_rows)};
            const cuuint32_t estr[2] = {1, 1};
            cr = enc(&e.map, dt, 2, const_cast<void*>(A), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        }
        if (cr != CUDA_SUCCESS) return -3;
        e.ptr = A;
        e.M = M;
        e.K = K;
        e.a_rows = a_rows;
        e.kps = kps;
        e.dt = DT;
        e.valid = 1;
        mp = &e.map;
    }

    TcArgs args;
    args.packed = static_cast<const uint8_t*>(packed);
    args.Y = Y;
    args.status = ctx.status;
    args.M = M;
    args.N = N;
    args.K = K;
    args.group = group;
    args.kblocks = blocks_k(K);
    args.splits = plan.split_k;
    args.a_stages = plan.stages;
    args.w_stages = plan.w_stages;
    args.a_rows = a_rows;
    args.kps = kps;
    args.a_2d = a_2d ? 1 : 0;
    args.slice_rows = tc_slice_rows(plan.split_k);
    args.flags = plan.prefetch_weights ? kFlagPrefetchW : 0;
    const TcLayout L = tc_layout(BM, M, group, plan.split_k, plan.stages, plan.w_stages);
    // This rank's own partials (all slices) are written to the start of the rings before
    // they are pushed; the receive area for the peers' partials follows the rings.
    if (plan.split_k > 1 && L.part_bytes > L.recv_off) return -2;
    if (plan.w_stages % tc_stage_multiple(BM, IL, NWG) != 0) return -2;
    if (plan.stages % tc_a_stage_multiple(BM, IL) != 0) return -2;
    args.a_stage_bytes = L.a_stage;
    args.w_stage_bytes = L.w_stage;
    args.w_off = L.w_off;
    args.recv_off = L.recv_off;
    args.timeout_ns = timeout_ns ? timeout_ns : ctx.timeout_ns;
    args.epi = epi;

    const size_t smem = L.smem;
    if (smem > static_cast<size_t>(ctx.max_smem_optin)) return -2;
    auto kern = w4a16_tc_kernel<BM, NWG, DT, DQ, IL, PROBE>;
    {   // raise the dynamic shared-memory limit once per device (not a stream operation,
        // but kept out of the steady state so that launches can be graph-captured cheaply)
        static std::mutex mu;
        static size_t configured[64] = {};  // per instantiation (template statics)
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
    cfg.gridDim = dim3(static_cast<unsigned>(plan.split_k), static_cast<unsigned>(tiles_n(N)),
                       static_cast<unsigned>((M + BM - 1) / BM));
    cfg.blockDim = dim3(32 * TcShape<BM, IL, NWG>::kDq0 + 128 * NWG, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int nattr = 0;
    if (plan.split_k > 1) {
        attr[nattr].id = cudaLaunchAttributeClusterDimension;
        attr[nattr].val.clusterDim.x = static_cast<unsigned>(plan.split_k);
        attr[nattr].val.clusterDim.y = 1;
        attr[nattr].val.clusterDim.z = 1;
        ++nattr;
    }
    if (plan.pdl) {
        attr[nattr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[nattr].val.programmaticStreamSerializationAllowed = 1;
        ++nattr;
    }
    cfg.attrs = attr;
    cfg.numAttrs = nattr;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, *mp, args);
    return e == cudaSuccess ? 0 : -3;
}

}  // namespace

int tc_a_rows(int tile_m, int M) {
    if (tile_m > 16) return tile_m;
    return M <= 8 ? 8 : 16;  // rows past M are zero-filled by the TMA
}

int tc_blocks_per_stage(int tile_m) { return tile_m <= 32 ? 2 : 1; }

TcLayout tc_layout(int tile_m, int M, int group, int split_k, int a_stages, int w_stages) {
    const int kps = tc_blocks_per_stage(tile_m);
    TcLayout L;
    // 2*kps chunks of 64 K x a_rows rows, 128 bytes per row: a multiple of 1024 bytes, so
    // every A stage keeps the alignment of the 128-byte swizzle pattern
    L.a_stage = static_cast<uint32_t>(2 * kps * tc_a_rows(tile_m, M)) * 128u;
    L.w_stage = (static_cast<uint32_t>(kps) * block_bytes(group, true) + 127u) & ~127u;
    L.w_off = static_cast<uint32_t>(a_stages) * L.a_stage;
    L.recv_off = (L.w_off + static_cast<uint32_t>(w_stages) * L.w_stage + 127u) & ~127u;
    const int slice = tc_slice_rows(split_k);
    L.part_bytes = split_k > 1 ? static_cast<uint32_t>(split_k * tile_m * slice * 4) : 0u;
    L.recv_bytes = split_k > 1 ? static_cast<uint32_t>((split_k - 1) * tile_m * slice * 4) : 0u;
    // + the control block + slack for aligning the dynamic shared base to 1024 bytes
    L.smem = static_cast<size_t>(L.recv_off) + L.recv_bytes + kCtrlBytes + 1024;
    return L;
}

int tc_a_stage_multiple(int tile_m, bool whole_blocks) {
    static_assert(TcShape<64, true, 4>::kSSteps == 2 && TcShape<128, true, 4>::kSSteps == 2,
                  "whole-block 64- and 128-row tiles: two issuers take alternate A stages");
    return (tile_m == 64 || tile_m == 128) && whole_blocks ? 2 : 1;
}

int tc_stage_multiple(int tile_m, bool whole_blocks, int nwg) {
    if (!whole_blocks) return 1;  // every warpgroup reads every stage
    const int kps = tc_blocks_per_stage(tile_m);
    return nwg > kps ? nwg / kps : 1;
}

int launch_tc_gemm(const DeviceCtx& ctx, const void* A, const void* packed, int M, int N,
                   int K, int group, int dtype, void* Y, const GemmPlan& plan,
                   const EpilogueArgs& epi, cudaStream_t stream) {
#define W4G_TC_CASE(BMV, NWGV)                                                            \
    case BMV:                                                                            \
        return dtype == 0                                                                \
                   ? launch_tc_instance<BMV, NWGV, 0>(ctx, A, packed, M, N, K, group, Y, \
                                                      plan, epi, stream)                 \
                   : launch_tc_instance<BMV, NWGV, 1>(ctx, A, packed, M, N, K, group, Y, \
                                                      plan, epi, stream);
    if (plan.dequant == 1) {  // the table unpack: decode tiles only
        switch (plan.tile_m) {
            case 16:
                return dtype == 0 ? launch_tc_instance<16, W4A16_SMALL_TILE_WG, 0, kDqLut>(
                                        ctx, A, packed, M, N, K, group, Y, plan, epi, stream)
                                  : launch_tc_instance<16, W4A16_SMALL_TILE_WG, 1, kDqLut>(
                                        ctx, A, packed, M, N, K, group, Y, plan, epi, stream);
            case 32:
                return dtype == 0 ? launch_tc_instance<32, W4A16_SMALL_TILE_WG, 0, kDqLut>(
                                        ctx, A, packed, M, N, K, group, Y, plan, epi, stream)
                                  : launch_tc_instance<32, W4A16_SMALL_TILE_WG, 1, kDqLut>(
                                        ctx, A, packed, M, N, K, group, Y, plan, epi, stream);
            default:
                return -2;
        }
    }
    if (plan.dequant == 2) {  // integer operand: 16-row tiles, groups of 128
        if (plan.tile_m != 16 || group != 128) return -2;
        return dtype == 0 ? launch_tc_instance<16, 2, 0, kDqInt>(ctx, A, packed, M, N, K, group,
                                                                Y, plan, epi, stream)
                          : launch_tc_instance<16, 2, 1, kDqInt>(ctx, A, packed, M, N, K, group,
                                                                Y, plan, epi, stream);
    }
#define W4G_TC_IL(BMV, NWGV)                                                               \
    return dtype == 0 ? launch_tc_instance<BMV, NWGV, 0, kDqMagic, true>(                   \
                            ctx, A, packed, M, N, K, group, Y, plan, epi, stream)           \
                      : launch_tc_instance<BMV, NWGV, 1, kDqMagic, true>(                   \
                            ctx, A, packed, M, N, K, group, Y, plan, epi, stream);
    if (plan.whole_blocks && plan.tile_m == 128 && plan.nwg == 4) { W4G_TC_IL(128, 4) }
    if (plan.whole_blocks && plan.tile_m == 64 && plan.nwg == 4) { W4G_TC_IL(64, 4) }
    if (plan.nwg == 4) {  // shared-block tiles with four warpgroups
        switch (plan.tile_m) {
            W4G_TC_CASE(256, 4)
            default:
                return -2;
        }
    }
    switch (plan.tile_m) {
        W4G_TC_CASE(16, W4A16_SMALL_TILE_WG)
        W4G_TC_CASE(32, W4A16_SMALL_TILE_WG)
        W4G_TC_CASE(64, 2)
        W4G_TC_CASE(128, 2)
        W4G_TC_CASE(256, 2)
        default:
            return -2;
    }
#undef W4G_TC_CASE
#undef W4G_TC_IL
}

int launch_tc_splitk_probe(const DeviceCtx& ctx, const void* A, const void* packed, int M,
                           int N, int K, int group, int dtype, void* Y, const GemmPlan& plan,
                           uint64_t timeout_ns, cudaStream_t stream) {
    if (plan.tile_m != 16 || plan.split_k < 2) return -2;
    const EpilogueArgs none{nullptr, nullptr, kActNone};
    return dtype == 0
               ? launch_tc_instance<16, W4A16_SMALL_TILE_WG, 0, kDqMagic, true, true>(
                     ctx, A, packed, M, N, K, group, Y, plan, none, stream, timeout_ns)
               : launch_tc_instance<16, W4A16_SMALL_TILE_WG, 1, kDqMagic, true, true>(
                     ctx, A, packed, M, N, K, group, Y, plan, none, stream, timeout_ns);
}

}  // namespace w4g
