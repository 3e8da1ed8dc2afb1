// layout.cuh -- the packed weight layout (version 1) shared by the library's kernels.
//
// The buffer is a 256-byte header followed by NB = ceil(N/64) n-blocks of KT = ceil(K/128)
// self-contained chunks.  Chunk (b, t) covers columns [64b, 64b+64) and rows [128t, 128t+128):
//   codes  4096 B: 64 column-rows x 64 B; row r (column 64b+r) holds 128 consecutive k as 16
//          uint32 words; word w holds k = 128t + 8w + kSlotK[j] in nibble slot j.
//   meta   (128/g) x 160 B: per group, 64 scales (fp16 or bf16) then 64 zero nibbles, in lane order
//          (position p = 8*(r%8) + 2*(r/16) + (r/8)%2 holds column-row r).
//
// Why this shape (GB300 reasoning, not taken from any page):
//  - n-blocks are independent and contiguous, so repack can run one n-range at a time and
//    produce identical bytes (the property the CPU plugin's n-block repack relies on).
//  - a column's 128 k-values are one 64-byte run, so 4 lanes x 16 B read one row-run and a
//    warp's 32 x 16 B vector load covers 8 column-rows: fully coalesced 512-byte requests for
//    the decode kernel, and contiguous 4 KB pieces for bulk copies.
//  - the slot order {0,2,4,6,1,3,5,7} makes the mask-and-or conversion of a word's nibbles
//    to fp16 (code OR'd into the mantissa of 1024.0) yield consecutive-k pairs in half2
//    registers: (w & 0x000F000F) holds k+0, k+1; (w & 0x00F000F0) holds k+2, k+3 (scaled by
//    16); the same on (w >> 8) gives k+4..k+7.
//  - meta in lane order lets a decode lane fetch all eight scales of its rows with one 16-byte
//    load and its eight zeros with one 4-byte load.
#pragma once
#include <cstdint>

namespace w4a16 {

constexpr uint32_t kMagic = 0x36314134u;
constexpr uint32_t kLayoutVersion = 1;
constexpr int kHeaderBytes = 256;
constexpr int kBlockN = 64;        // columns per n-block
constexpr int kTileK = 128;        // rows of K per chunk
constexpr int kCodeBytes = 4096;   // 64 rows x 64 bytes
constexpr int kRowBytes = 64;      // one column's 128 codes
constexpr int kGroupMetaBytes = 160;
constexpr int kScaleBytes = 128;   // 64 fp16 scales of one group

// nibble slot j of a code word -> k offset inside the word's 8 rows
__host__ __device__ constexpr int slot_k(int j) { return (j < 4) ? 2 * j : 2 * (j - 4) + 1; }

__host__ __device__ inline int chunk_bytes(int g) { return kCodeBytes + (kTileK / g) * kGroupMetaBytes; }
__host__ __device__ inline int num_nblocks(int N) { return (N + kBlockN - 1) / kBlockN; }
__host__ __device__ inline int num_ktiles(int K) { return (K + kTileK - 1) / kTileK; }

// bytes of a packed buffer of a K x N layer with layout group size g (header included)
__host__ __device__ inline long long packed_extent(int K, int N, int g) {
  return kHeaderBytes + (long long)num_nblocks(N) * num_ktiles(K) * chunk_bytes(g);
}

// lane-order position of column-row r (0..63) inside a group's meta
__host__ __device__ inline int meta_pos(int r) { return 8 * (r % 8) + 2 * (r / 16) + (r / 8) % 2; }

// dtype: element type of x, the scales, the weights and y -- 0 fp16, 1 bf16 (the codes and the
// zero nibbles do not depend on it).  The rest of the 256 bytes is zero.
struct Header {
  uint32_t magic, version;
  int32_t K, N, g, dtype;
};
constexpr int kDtypeF16 = 0;
constexpr int kDtypeBf16 = 1;

}  // namespace w4a16
