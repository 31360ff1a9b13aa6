"""The measured premise of the W4A8 GEMM's tensor path (GPU).

"W4A8量化计算优化" §3.2 feeds the int8 weights to an int8 x int8 -> int32 tensor-core MMA.
On sm_103a the tcgen05 family has no int8 kind (tests/test_toolchain_mma_kinds.py), and
this test measures the other two routes: the int8 mma.sync, which runs no faster than
dp4a on the CUDA cores, and the f16 mma.sync, which runs several times faster.  The W4A8
GEMM therefore carries its int8 values, exactly, through the f16 mma.sync.  The probe
is a plain throughput loop (four independent accumulators per warp, eight 256-thread CTAs
per SM), built with nvcc and run once; it prints the rates it measured.
"""
import os
import re
import shutil
import subprocess
import tempfile

import pytest
import torch

pytestmark = pytest.mark.gpu

NVCC = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"

_SRC = r"""
#include <cstdio>
#include <cstdint>
#include <cuda_runtime.h>
constexpr int ITER = 1024;
__global__ void mma_s8(const uint32_t* in, int* out) {
    uint32_t a0 = in[threadIdx.x & 7], a1 = a0 ^ 1, a2 = a0 ^ 2, a3 = a0 ^ 3, b0 = a0 ^ 4, b1 = a0 ^ 5;
    int c[4][4] = {};
    for (int i = 0; i < ITER; ++i) {
#pragma unroll
        for (int j = 0; j < 4; ++j)
            asm volatile("mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, "
                         "{%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
                         : "+r"(c[j][0]), "+r"(c[j][1]), "+r"(c[j][2]), "+r"(c[j][3])
                         : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
    int s = 0;
    for (int j = 0; j < 4; ++j) s += c[j][0] + c[j][1] + c[j][2] + c[j][3];
    out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}
__global__ void mma_f16(const uint32_t* in, int* out) {
    uint32_t a0 = in[threadIdx.x & 7] & 0x3c003c00u, a1 = a0, a2 = a0, a3 = a0, b0 = a0, b1 = a0;
    float c[4][4] = {};
    for (int i = 0; i < ITER; ++i) {
#pragma unroll
        for (int j = 0; j < 4; ++j)
            asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, "
                         "{%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
                         : "+f"(c[j][0]), "+f"(c[j][1]), "+f"(c[j][2]), "+f"(c[j][3])
                         : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
    float s = 0;
    for (int j = 0; j < 4; ++j) s += c[j][0] + c[j][1] + c[j][2] + c[j][3];
    out[blockIdx.x * blockDim.x + threadIdx.x] = (int)s;
}
__global__ void dp4a_k(const uint32_t* in, int* out) {
    int a = (int)in[threadIdx.x & 7];
    int c[8] = {};
    for (int i = 0; i < ITER; ++i) {
#pragma unroll
        for (int j = 0; j < 8; ++j) c[j] = __dp4a(a + j, a ^ i, c[j]);
    }
    int s = 0;
    for (int j = 0; j < 8; ++j) s += c[j];
    out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}
int main() {
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
    const int blocks = sms * 8, threads = 256;
    uint32_t* in; int* out;
    if (cudaMalloc(&in, 64) != cudaSuccess || cudaMalloc(&out, sizeof(int) * blocks * threads) != cudaSuccess) return 2;
    uint32_t h[16] = {0x01020304u, 0x05060708u, 0x7f7f0101u, 0x80818283u, 3, 5, 7, 9};
    cudaMemcpy(in, h, 64, cudaMemcpyHostToDevice);
    cudaEvent_t e0, e1; cudaEventCreate(&e0); cudaEventCreate(&e1);
    const double warps = blocks * threads / 32.0;
    const char* names[3] = {"mma_s8", "mma_f16", "dp4a"};
    for (int kind = 0; kind < 3; ++kind) {
        float ms = 0;
        for (int rep = 0; rep < 2; ++rep) {
            cudaEventRecord(e0);
            if (kind == 0) mma_s8<<<blocks, threads>>>(in, out);
            else if (kind == 1) mma_f16<<<blocks, threads>>>(in, out);
            else dp4a_k<<<blocks, threads>>>(in, out);
            cudaEventRecord(e1);
            cudaEventSynchronize(e1);
            cudaEventElapsedTime(&ms, e0, e1);
        }
        const double macs = kind == 0 ? warps * ITER * 4 * 16.0 * 8 * 32
                          : kind == 1 ? warps * ITER * 4 * 16.0 * 8 * 16
                                      : blocks * (double)threads * ITER * 8 * 4;
        printf("%s %.3f\n", names[kind], macs / ms / 1e9);
    }
    return cudaGetLastError() == cudaSuccess ? 0 : 1;
}
"""


def test_f16_mma_outruns_the_int8_routes():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    with tempfile.TemporaryDirectory() as d:
        src, exe = os.path.join(d, "rates.cu"), os.path.join(d, "rates")
        open(src, "w").write(_SRC)
        subprocess.run([NVCC, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-o", exe, src],
                       check=True, capture_output=True)
        r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    rate = {m.group(1): float(m.group(2)) for m in re.finditer(r"(\w+) ([0-9.]+)", r.stdout)}
    print("T MAC/s:", rate)
    assert rate["mma_f16"] > 2.0 * rate["mma_s8"], rate
    assert rate["mma_f16"] > 2.0 * rate["dp4a"], rate
