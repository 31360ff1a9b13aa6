// Fused epilogue of the GEMM kernels ("量化开销对比" §6.2: accumulator x scale -> + bias ->
// store; §6.6: scale + bias, + residual / activation, in the same kernel).  Applied in
// fp32 to the finished fp32 sum (already multiplied by the per-channel factor):
//     y = act(v + bias[n]) + residual[m, n]
// act: 0 identity, 1 ReLU, 2 SiLU (v / (1 + exp(-v))).  The thread that writes Y[m, n]
// is the one that reads residual[m, n] (before it writes), so residual may be Y itself
// (in-place add).
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace w4g {

constexpr int kActNone = 0;
constexpr int kActRelu = 1;
constexpr int kActSilu = 2;

struct EpilogueArgs {
    const uint16_t* bias;      // dtype [N] or null
    const uint16_t* residual;  // dtype [M][N] or null
    int act;
};

template <int DT>
__device__ __forceinline__ float dtype_to_f32(uint16_t bits) {
    if constexpr (DT == 0) return __half2float(__ushort_as_half(bits));
    else return __bfloat162float(__ushort_as_bfloat16(bits));
}

// SiLU through the identity v * sigmoid(v) = (v / 2) * (1 + tanh(v / 2)), with the
// hardware tanh approximation (tanh.approx.f32, relative error about 2^-11): one special-
// function operation per element instead of an exponential and a reciprocal.  Its error,
// at most |v| / 2 * 2^-11, is far inside the result's bound (1e-3 of the magnitude sum,
// which is at least |v|).
__device__ __forceinline__ float tanh_approx(float x) {
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float apply_activation(float v, int act) {
    if (act == kActRelu) return fmaxf(v, 0.0f);
    if (act == kActSilu) {
        const float h = 0.5f * v;
        return fmaf(h, tanh_approx(h), h);
    }
    return v;
}

// bias_n: the channel's bias as fp32 (0 when there is none).
template <int DT>
__device__ __forceinline__ float apply_epilogue(float v, float bias_n, const EpilogueArgs& e,
                                                size_t idx) {
    v = apply_activation(v + bias_n, e.act);
    if (e.residual) v += dtype_to_f32<DT>(e.residual[idx]);
    return v;
}

}  // namespace w4g
