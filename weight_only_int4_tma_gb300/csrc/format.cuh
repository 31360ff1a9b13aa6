// Packed-weight format shared by the repack, debug-dequant and GEMM kernels.
//
// Offline repack into the kernel's tile order ("量化开销对比" §6.4): the unit is a block
// of 128 output channels x 128 values of K.  Blocks of one channel tile are contiguous
// along K, so any K range of a tile is one contiguous byte range that a single bulk
// TMA copy moves into shared memory, scales and zeros included.
//
// Shapes that are not multiples of 128 are padded to whole blocks at repack time (zero
// scales and nibbles past N or K); the header keeps the logical N and K.
//
// Block layout (all offsets in bytes from the block start):
//   [0, 8192)           nibbles: chunk c (32 K values) x row r (128) x word w (4),
//                       16 bytes per (c, r).  A warp reading rows r..r+31 of one chunk
//                       touches 512 contiguous bytes: one conflict-free 128-bit
//                       shared-memory load per thread.
//   [8192, +G*256)      scales: group gi (G = 128/group per block) x row r, raw dtype
//                       bits, 2 bytes each.
//   [.., +G*64)         zeros (only if the blob has zeros): group gi x 64 bytes; row r's
//                       zero is nibble (r & 1) of byte r/2.
// Within a word the eight K values k0..k7 (K offset 8w + j inside the chunk) sit at
// nibble positions p(j) = 4*(j & 1) + (j >> 1): positions (0,4) hold (k0,k1),
// (1,5) hold (k2,k3), (2,6) hold (k4,k5), (3,7) hold (k6,k7).  Shifting the word right
// by 4*i and masking 0x000F000F therefore yields the pair (k_2i, k_2i+1) in the two
// 16-bit halves, ready for the exponent-injection unpack
// ("W4A16 GEMM 算子浅析" §"Marlin 与 CUTLASS 中的寄存器解包黑魔法").
#pragma once
#include <cstdint>

namespace w4g {

constexpr uint32_t kMagic = 0x4B503457u;  // "W4PK"
constexpr uint32_t kVersion = 1;
constexpr int kHeaderBytes = 128;
constexpr int kTileN = 128;               // output channels per block
constexpr int kTileK = 128;               // K values per block
constexpr int kChunkK = 32;               // K values per 16-byte chunk of one row
constexpr int kNibbleBytes = kTileN * kTileK / 2;  // 8192

constexpr uint32_t kFlagZeros = 1u;
constexpr uint32_t kFlagChannelScale = 2u;

struct PackedHeader {
    uint32_t magic;
    uint32_t version;
    int32_t N;
    int32_t K;
    int32_t group;
    int32_t dtype;
    uint32_t flags;
    uint32_t block_bytes;
    uint64_t body_offset;
    uint64_t cscale_offset;  // 0 when absent
    uint64_t total_bytes;
    uint32_t reserved[18];
};
static_assert(sizeof(PackedHeader) == kHeaderBytes, "header must be 128 bytes");

__host__ __device__ constexpr int groups_per_block(int group) { return kTileK / group; }
__host__ __device__ constexpr uint32_t scale_bytes(int group) {
    return static_cast<uint32_t>(groups_per_block(group)) * kTileN * 2u;
}
__host__ __device__ constexpr uint32_t zero_bytes(int group) {
    return static_cast<uint32_t>(groups_per_block(group)) * (kTileN / 2u);
}
__host__ __device__ constexpr uint32_t block_bytes(int group, bool zeros) {
    return kNibbleBytes + scale_bytes(group) + (zeros ? zero_bytes(group) : 0u);
}

// Blocks along N and K: the blob covers ceil(N/128) x ceil(K/128) blocks; positions past
// N or K hold zero scales (so the padded weights are exactly 0) and zero nibbles.
__host__ __device__ constexpr int tiles_n(int N) { return (N + kTileN - 1) / kTileN; }
__host__ __device__ constexpr int blocks_k(int K) { return (K + kTileK - 1) / kTileK; }

// Nibble position of K offset j (0..7) inside a packed word.
__host__ __device__ constexpr int nibble_pos(int j) { return 4 * (j & 1) + (j >> 1); }

// Device-side check of a blob header against the call's arguments: returns the flags,
// or -1 on any mismatch (wrong magic/version/shape/group/dtype/block size).
__device__ __forceinline__ int check_header(const PackedHeader* h, int N, int K, int group,
                                            int dtype) {
    if (h->magic != kMagic || h->version != kVersion || h->N != N || h->K != K ||
        h->group != group || h->dtype != dtype)
        return -1;
    const bool z = (h->flags & kFlagZeros) != 0;
    if (h->block_bytes != block_bytes(group, z) || h->body_offset != kHeaderBytes) return -1;
    return static_cast<int>(h->flags);
}

}  // namespace w4g
