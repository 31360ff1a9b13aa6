// Register-level unpack + dequant of one packed word (8 weights) into four 16-bit pairs.
//
// "W4A16 GEMM 算子浅析" §"Marlin 与 CUTLASS 中的寄存器解包黑魔法": OR-ing a nibble into
// the mantissa of the pattern 0x6400 (fp16 1024.0) gives the fp16 number 1024 + q with
// no integer-to-float conversion.  The page's printed mask 0x0F0F0F0F would leave two
// nibbles in one half; the per-half mask here is 0x000F000F, and the packed format puts
// the pair (k_2i, k_2i+1) at nibble positions (i, i+4) so that (x >> 4i) & 0x000F000F
// selects it.  bf16 uses 0x4300 (128.0), whose 7-bit mantissa also has unit spacing.
//
// The value must be ONE round-to-nearest-even of (q - z) * s ("计算流水线的核心哲学" step 2,
// W = (W_int4 - Zero) * Scale).  A single fma with a pre-rounded -(1024 + z) * s constant
// would round twice, so the pair is formed as
//     t = (1024 + q) - (1024 + z)   exact: an integer in [-15, 15]
//     w = t * s                     one rounding, to nearest even
// with sub.rn / mul.rn on packed pairs: one LOP3 + one SUB + one MUL per pair of weights.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

namespace w4g {

template <int DT>
struct Magic;
template <>
struct Magic<0> {  // fp16: 1024.0 in each half
    static constexpr uint32_t kPair = 0x64006400u;
};
template <>
struct Magic<1> {  // bf16: 128.0 in each half
    static constexpr uint32_t kPair = 0x43004300u;
};

__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;  // (a & b) | c
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

template <int DT>
__device__ __forceinline__ uint32_t sub_pair(uint32_t a, uint32_t b) {
    uint32_t d;
    if constexpr (DT == 0) {
        asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    } else {
        asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    }
    return d;
}

template <int DT>
__device__ __forceinline__ uint32_t mul_pair(uint32_t a, uint32_t b) {
    uint32_t d;
    if constexpr (DT == 0) {
        asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    } else {
        asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    }
    return d;
}

// Per-(group, row) constants: biased zero (1024 + z or 128 + z in both halves) and the
// scale in both halves.
template <int DT>
__device__ __forceinline__ uint32_t zero_pair(uint32_t z) {
    return Magic<DT>::kPair | (z * 0x00010001u);
}
__device__ __forceinline__ uint32_t scale_pair(uint32_t sbits) {
    return sbits * 0x00010001u;
}

// x: one packed word (see format.cuh).  out[i] = (w[k_2i], w[k_2i+1]) as a 16-bit pair.
template <int DT>
__device__ __forceinline__ void dequant_word(uint32_t x, uint32_t zp, uint32_t sp,
                                             uint32_t* out) {
    constexpr uint32_t kMask = 0x000F000Fu;
    constexpr uint32_t kM = Magic<DT>::kPair;
    const uint32_t t0 = lop3_and_or(x, kMask, kM);
    const uint32_t t1 = lop3_and_or(x >> 4, kMask, kM);
    const uint32_t t2 = lop3_and_or(x >> 8, kMask, kM);
    const uint32_t t3 = lop3_and_or(x >> 12, kMask, kM);
    out[0] = mul_pair<DT>(sub_pair<DT>(t0, zp), sp);
    out[1] = mul_pair<DT>(sub_pair<DT>(t1, zp), sp);
    out[2] = mul_pair<DT>(sub_pair<DT>(t2, zp), sp);
    out[3] = mul_pair<DT>(sub_pair<DT>(t3, zp), sp);
}

// fp16 only, two shifts fewer per word: the pairs at nibble positions (1,5) and (3,7)
// are masked in place (0x00F000F0), which puts q in mantissa bits 4..7, i.e. the fp16
// number 1024 + 16 q.  Then (1024 + 16q) - (1024 + 16z) = 16 (q - z) exactly, and
// multiplying by s/16 rounds once to rn((q - z) s) -- provided s/16 is itself exact
// (checked per group by the caller with f16_div16_exact()).
__device__ __forceinline__ void dequant_word_f16_x16(uint32_t x, uint32_t zp, uint32_t sp,
                                                     uint32_t zp16, uint32_t sp16,
                                                     uint32_t* out) {
    constexpr uint32_t kM = Magic<0>::kPair;
    const uint32_t y = x >> 8;
    const uint32_t t0 = lop3_and_or(x, 0x000F000Fu, kM);
    const uint32_t t1 = lop3_and_or(x, 0x00F000F0u, kM);
    const uint32_t t2 = lop3_and_or(y, 0x000F000Fu, kM);
    const uint32_t t3 = lop3_and_or(y, 0x00F000F0u, kM);
    out[0] = mul_pair<0>(sub_pair<0>(t0, zp), sp);
    out[1] = mul_pair<0>(sub_pair<0>(t1, zp16), sp16);
    out[2] = mul_pair<0>(sub_pair<0>(t2, zp), sp);
    out[3] = mul_pair<0>(sub_pair<0>(t3, zp16), sp16);
}

// (1024 + 16 z) in both fp16 halves.
__device__ __forceinline__ uint32_t zero_pair_x16(uint32_t z) {
    return Magic<0>::kPair | ((z << 4) * 0x00010001u);
}

// s/16 in both halves (a power-of-two scaling: exact unless it leaves the normal range).
__device__ __forceinline__ uint32_t scale_pair_div16(uint32_t sp) {
    return mul_pair<0>(sp, 0x2C002C00u);  // x 0.0625
}

// True when s/16 * 16 == s bit for bit, i.e. the division by 16 lost nothing.
__device__ __forceinline__ bool f16_div16_exact(uint32_t sp, uint32_t sp16) {
    return mul_pair<0>(sp16, 0x4C004C00u) == sp;  // x 16
}

// ---- integer-operand variant (the MMA takes the exact integers q - z; the group scale
// multiplies each block's fp32 partial sum afterwards) ---------------------------------

template <int DT>
__device__ __forceinline__ uint32_t fma_pair(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    if constexpr (DT == 0) {
        asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    } else {
        asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    }
    return d;
}

// out[i] = (q_2i - z, q_2i+1 - z), exact small integers in the activation dtype.
// bf16: the four pairs are shifted down and biased like dequant_word, without the scale.
// fp16: the pairs at nibble positions (1,5) and (3,7) are masked in place (1024 + 16 q)
// and fma'd with 1/16 and -(64 + z): (64 + q) - (64 + z), exact inside the fma.
template <int DT>
__device__ __forceinline__ void int_word(uint32_t x, uint32_t zp, uint32_t nz64,
                                         uint32_t* out) {
    constexpr uint32_t kM = Magic<DT>::kPair;
    if constexpr (DT == 0) {
        const uint32_t y = x >> 8;
        out[0] = sub_pair<0>(lop3_and_or(x, 0x000F000Fu, kM), zp);
        out[1] = fma_pair<0>(lop3_and_or(x, 0x00F000F0u, kM), 0x2C002C00u, nz64);
        out[2] = sub_pair<0>(lop3_and_or(y, 0x000F000Fu, kM), zp);
        out[3] = fma_pair<0>(lop3_and_or(y, 0x00F000F0u, kM), 0x2C002C00u, nz64);
    } else {
        out[0] = sub_pair<1>(lop3_and_or(x, 0x000F000Fu, kM), zp);
        out[1] = sub_pair<1>(lop3_and_or(x >> 4, 0x000F000Fu, kM), zp);
        out[2] = sub_pair<1>(lop3_and_or(x >> 8, 0x000F000Fu, kM), zp);
        out[3] = sub_pair<1>(lop3_and_or(x >> 12, 0x000F000Fu, kM), zp);
    }
}

// -(64 + z) in both fp16 halves (exact).
__device__ __forceinline__ uint32_t neg64_pair(uint32_t z) {
    return static_cast<uint32_t>(__half_as_ushort(__float2half_rn(-(64.0f + static_cast<float>(z))))) *
           0x00010001u;
}

// ---- table variant ("量化开销对比" §6.3: nibble -> value through a 16-entry table in
// shared memory, then the group's zero and scale) ----------------------------------------

// Bits of the small integer q (0..15) in the activation dtype (exact).
template <int DT>
__device__ __forceinline__ uint16_t value_bits(int q) {
    if constexpr (DT == 0) return __half_as_ushort(__float2half_rn(static_cast<float>(q)));
    else return __bfloat16_as_ushort(__float2bfloat16_rn(static_cast<float>(q)));
}

// z in both halves, read from the table.
__device__ __forceinline__ uint32_t lut_zero_pair(const uint16_t* lut, uint32_t z) {
    return static_cast<uint32_t>(lut[z]) * 0x00010001u;
}

// Same output as dequant_word: each pair (q_2i, q_2i+1) is looked up in the table, then
// (q - z) is formed exactly and multiplied by s with one rounding.
template <int DT>
__device__ __forceinline__ void dequant_word_lut(uint32_t x, const uint16_t* lut, uint32_t zp,
                                                 uint32_t sp, uint32_t* out) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t lo = (x >> (4 * i)) & 0xFu;
        const uint32_t hi = (x >> (4 * i + 16)) & 0xFu;
        const uint32_t t = static_cast<uint32_t>(lut[lo]) | (static_cast<uint32_t>(lut[hi]) << 16);
        out[i] = mul_pair<DT>(sub_pair<DT>(t, zp), sp);
    }
}

}  // namespace w4g
