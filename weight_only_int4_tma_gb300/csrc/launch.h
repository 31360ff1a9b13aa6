// Internal host-side interface between the C-ABI layer (api.cu) and the kernel units.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "epilogue.cuh"

namespace w4g {

// Per-device state, created once per device on first use.
struct DeviceCtx {
    int device;
    int num_sms;
    int max_smem_optin;     // bytes of dynamic shared memory a CTA may opt into
    int* status;            // device address of this device's status word
    uint64_t timeout_ns;    // limit of every bounded in-kernel wait
};

struct GemmPlan {
    int kernel;   // 1 = tcgen05, 2 = SIMT
    int tile_m;   // activation rows per tile (tcgen05 kernel); channels per unit (SIMT)
    int split_k;  // K slices (cluster size for the tcgen05 kernel)
    int stages;   // tcgen05 kernel: depth of the A ring
    int w_stages; // tcgen05 kernel: depth of the weight ring
    bool pdl;               // launch with programmatic dependent launch
    bool prefetch_weights;  // read the packed blob before the dependency wait
    int dequant;            // tensor-core decode tiles: 0 exponent injection, 1 the
                            // 16-entry table, 2 integer operand + fp32 group rescale
    bool whole_blocks;      // tensor-core kernel: each dequant warpgroup unpacks whole blocks
    int nwg;                // tensor-core kernel: dequant warpgroups
};

// Launchers return a w4a16_status code.
int launch_repack(const DeviceCtx& ctx, const uint32_t* qweight, const void* scales,
                  const uint32_t* qzeros, const void* cscale, int N, int K, int group,
                  int dtype, void* packed, cudaStream_t stream);

int launch_dequant_debug(const DeviceCtx& ctx, const void* packed, int N, int K, int group,
                         int dtype, void* W_out, cudaStream_t stream);

int launch_tc_gemm(const DeviceCtx& ctx, const void* A, const void* packed, int M, int N,
                   int K, int group, int dtype, void* Y, const GemmPlan& plan,
                   const EpilogueArgs& epi, cudaStream_t stream);

int launch_simt_gemm(const DeviceCtx& ctx, const void* A, const void* packed, int M, int N,
                     int K, int group, int dtype, void* Y, const GemmPlan& plan,
                     const EpilogueArgs& epi, cudaStream_t stream);

int launch_timeout_probe(const DeviceCtx& ctx, uint64_t limit_ns, cudaStream_t stream);

// The tensor-core kernel (16-row tiles, split-K) with cluster rank 0 pushing none of its
// partials, every bounded wait limited to timeout_ns: a failure-path check of the split-K
// exchange.
int launch_tc_splitk_probe(const DeviceCtx& ctx, const void* A, const void* packed, int M,
                           int N, int K, int group, int dtype, void* Y, const GemmPlan& plan,
                           uint64_t timeout_ns, cudaStream_t stream);

// W4A8 path (w4a8.cu): blob size, repack, int8 debug expansion, per-row activation
// quantisation and the dp4a GEMM (M <= 16; returns -2 beyond).
size_t w4a8_blob_bytes(int N, int K);
int launch_w4a8_repack(const DeviceCtx& ctx, const uint32_t* qweight, const uint8_t* s_u8,
                       const uint8_t* off, const float* s_w, int N, int K, void* packed,
                       cudaStream_t stream);
int launch_w4a8_dequant_debug(const DeviceCtx& ctx, const void* packed, int N, int K,
                              void* W_out, cudaStream_t stream);
int launch_w4a8_quantize(const DeviceCtx& ctx, const void* A, int M, int K, int dtype,
                         int8_t* A_i8, float* s_a, cudaStream_t stream);
int launch_w4a8_gemm(const DeviceCtx& ctx, const int8_t* A_i8, const float* s_a,
                     const void* packed, int M, int N, int K, int dtype, void* Y,
                     cudaStream_t stream);

// MX block-scaled decode GEMM (mxfp.cu): blob size, repack, GEMM (M <= 16; -2 beyond).
size_t mx_blob_bytes(int N, int K);
int launch_mx_repack(const DeviceCtx& ctx, const uint8_t* w_codes, const uint8_t* w_scales,
                     int N, int K, void* packed, cudaStream_t stream);
int launch_mx_gemm(const DeviceCtx& ctx, const uint8_t* a_codes, const uint8_t* a_scales,
                   const void* packed, int M, int N, int K, int dtype, void* Y,
                   cudaStream_t stream);

// Rows of A staged per 64-K chunk (8 or 16 for decode tiles, else the tile height).
int tc_a_rows(int tile_m, int M);
// 128-K weight blocks per ring stage (one bulk copy each stage).
int tc_blocks_per_stage(int tile_m);
// Channels of a 128-channel tile owned by each cluster rank under split-K: ceil(128 /
// split_k) rounded up to a multiple of 4, so that every rank's slice of the partials is
// read and stored 4 channels at a time (the last rank may own fewer).
inline int tc_slice_rows(int split_k) { return ((128 + split_k - 1) / split_k + 3) & ~3; }
// Deepest ring of either kind (the control block holds 16 barriers per ring).
constexpr int kTcMaxStages = 16;
// Shared-memory layout of the tcgen05 kernel: [A ring][weight ring][split-K receive
// area][control block], offsets from the 1024-byte aligned dynamic shared base.
struct TcLayout {
    uint32_t a_stage;     // bytes of one A stage
    uint32_t w_stage;     // bytes of one weight stage
    uint32_t w_off;       // weight ring
    uint32_t recv_off;    // receive area (end of the rings)
    uint32_t recv_bytes;  // receive area: one slice per other rank (0 without split-K)
    uint32_t part_bytes;  // this rank's partials of every slice, staged at the start of
                          // the rings before they are pushed (0 without split-K)
    size_t smem;          // dynamic shared memory to request
};
TcLayout tc_layout(int tile_m, int M, int group, int split_k, int a_stages, int w_stages);
// The weight ring depth must be a multiple of this (with whole blocks per warpgroup, each
// dequant warpgroup then reads a fixed subset of the weight slots and passes every phase
// of their barriers).
int tc_stage_multiple(int tile_m, bool whole_blocks, int nwg);
// The A ring depth must be a multiple of this (2 where two MMA issuers take every other
// stage, so that each A slot has one waiting issuer).
int tc_a_stage_multiple(int tile_m, bool whole_blocks);

}  // namespace w4g
