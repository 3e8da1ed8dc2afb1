// repack.cu -- one-time, integer-exact repack of AWQ tensors into the packed layout.
//
// Input (vLLM walkthrough "Carga de capas cuantizadas: AWQ / GPTQ / Marlin / fp8", section
// "Flujo de datos"): qweight int32 [K][N/8] and qzeros int32 [K/g][N/8], both packed along the
// output dimension; scales fp16 [K/g][N] (bf16 for a bf16 layer: the scales are copied as
// 16-bit patterns, so only the header's dtype word differs).  AWQ puts column 8c + {0,2,4,6,1,3,5,7}[j] of a word
// in nibble slot j (the "non-standard packing order along the output dimension" of section
// "Motivacion de diseno").  This is the analogue of process_weights_after_loading: done once,
// on the device, with no int32 expansion of the codes (vllm-omni commit "cpu_int4: repack
// weights in n-blocks, to bound the load-time peak" measured that transient at 8x the packed
// size).  A CTA writes the chunks of four consecutive n-blocks of one k-tile, reading each AWQ row
// as one 128-byte segment; chunks are self-contained, so any n-range can be repacked on its own.
#include <cuda_runtime.h>

#include "bounds.cuh"
#include "kernels.h"
#include "layout.cuh"
#include "nibble.cuh"

namespace w4a16 {
namespace {

// column offset inside an AWQ word -> its nibble slot (inverse of {0,2,4,6,1,3,5,7})
__device__ __forceinline__ int awq_slot_of_col(int c) { return (c & 1) ? 4 + (c >> 1) : (c >> 1); }

// lane-order position p -> column-row r (inverse of meta_pos)
__device__ __forceinline__ int meta_row(int p) { return 16 * ((p % 8) / 2) + 8 * (p % 2) + p / 8; }

constexpr int kRepackBlocks = 4;  // n-blocks per CTA: 32 AWQ words = 128 contiguous bytes of a row
constexpr int kRepackThreads = 256;

// XOR applied to the code-word index w of column-row r of n-block bl in the shared output tile, so
// that the transposing threads' stores (32 lanes: 4 n-blocks x 8 words of 8 columns) and the
// copy-out's reads both hit distinct banks.
__device__ __forceinline__ int out_swizzle(int bl, int r) { return ((r >> 5) & 1) | (bl << 1); }

// One CTA: kRepackBlocks consecutive n-blocks b0 + 4 blockIdx.x + bl (those below b1) of k-tile t.
__global__ void __launch_bounds__(kRepackThreads) repack_kernel(
    const int32_t *__restrict__ qweight, int64_t ldq, const int32_t *__restrict__ qzeros,
    int64_t ldz, const uint16_t *__restrict__ scales, int64_t lds, int K, int N, int g, int gsrc, int dtype,
    int n0, int n1, int b0, int b1, int KT, uint8_t *__restrict__ packed, int *err) {
  const int bfirst = b0 + kRepackBlocks * blockIdx.x;  // first n-block of this CTA
  const int t = blockIdx.y;                            // k-tile
  const int kb = t * kTileK;
  const int CB = chunk_bytes(g);
  // extents of the source slices (columns [n0, n1) at their row strides) and of `packed`, in bytes
  const int Gs = K / gsrc;
  const long long wq = (n1 - n0) / 8;
  const long long qext = 4 * ((K - 1) * ldq + wq), zext = 4 * ((Gs - 1) * ldz + wq);
  const long long sext = 2 * ((Gs - 1) * lds + (n1 - n0)), pext = packed_extent(K, N, g);

  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x < kHeaderBytes / 4) {
    uint32_t v = 0;
    switch (threadIdx.x) {
      case 0: v = kMagic; break;
      case 1: v = kLayoutVersion; break;
      case 2: v = (uint32_t)K; break;
      case 3: v = (uint32_t)N; break;
      case 4: v = (uint32_t)g; break;
      case 5: v = (uint32_t)dtype; break;
      default: v = 0;
    }
    if (in_extent(reinterpret_cast<uint32_t *>(packed) + threadIdx.x, 4, packed, pext, err))
      reinterpret_cast<uint32_t *>(packed)[threadIdx.x] = v;
  }

  // The code words.  Row r of n-block b (column 64 b + r), word w holds k = kb + 8w + slot_k(j) in
  // slot j.  A thread takes kUnits (word-column c, k-octet w) units of the CTA's 32 x 16, c
  // fastest, and loads the 8 AWQ words of rows kb + 8w + slot_k(j) (j = 0..7) of word-column c --
  // 8 k x 8 columns of nibbles -- straight into registers (a warp's load is one row's 128
  // contiguous bytes; rows past K, columns past N or past the last n-block read as 0), every word
  // requested before any is used.  Transposed in registers, word p is the code word of the column
  // in AWQ slot p.
  constexpr int kW = 8 * kRepackBlocks;  // AWQ words of a row in this CTA
  constexpr int kUnits = kW * 16 / kRepackThreads;
  static_assert((kW * 16) % kRepackThreads == 0 && (kBlockN * 16) % kRepackThreads == 0 &&
                    (kRepackBlocks * 4 * kBlockN) % kRepackThreads == 0,
                "the unrolled loads, scale loads and code copy-out give every thread the same count");
  const int gpc = kTileK / g;            // groups per chunk
  const int G = K / g;
  __shared__ uint32_t out[kRepackBlocks][kBlockN][17];  // code words per n-block (row stride 17)
  __shared__ uint32_t zin[4][kW];                       // [group of the chunk][AWQ zero word]
  uint32_t R[kUnits][8];
#pragma unroll
  for (int u = 0; u < kUnits; ++u) {
    const int i = (int)threadIdx.x + u * kRepackThreads, c = i % kW, w = i / kW;
    const int b = bfirst + c / 8, n = b * kBlockN + 8 * (c % 8);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int k = kb + 8 * w + slot_k(j);
      const int32_t *src = qweight + (int64_t)k * ldq + (n - n0) / 8;
      R[u][j] = (k < K && b < b1 && n < N && in_extent(src, 4, qweight, qext, err)) ? (uint32_t)__ldg(src) : 0u;
    }
  }
  // the scales of the CTA's n-blocks, requested with the codes (at most 4 groups per chunk)
  __shared__ uint16_t sin[kRepackBlocks][4][kBlockN];  // [n-block][group of the chunk][column]
#pragma unroll
  for (int u = 0; u < (kRepackBlocks * 4 * kBlockN) / kRepackThreads; ++u) {
    const int i = (int)threadIdx.x + u * kRepackThreads;
    const int bl = i / (4 * kBlockN), l = (i / kBlockN) % 4, r = i % kBlockN;
    if (l < gpc) {
      const int b = bfirst + bl, grp = t * gpc + l, n = b * kBlockN + r;
      const int sg = (grp * g) / gsrc;
      const uint16_t *src = scales + (int64_t)sg * lds + (n - n0);
      sin[bl][l][r] = (b < b1 && grp < G && n < N && in_extent(src, 2, scales, sext, err)) ? __ldg(src) : (uint16_t)0;
    }
  }
  if (threadIdx.x < gpc * kW) {
    const int l = threadIdx.x / kW, c = threadIdx.x % kW;
    const int grp = t * gpc + l, b = bfirst + c / 8, n = b * kBlockN + 8 * (c % 8);
    const int sg = (grp * g) / gsrc;
    const int32_t *src = qzeros + (int64_t)sg * ldz + (n - n0) / 8;
    zin[l][c] = (grp < G && b < b1 && n < N && in_extent(src, 4, qzeros, zext, err)) ? (uint32_t)__ldg(src) : 0u;
  }
#pragma unroll
  for (int u = 0; u < kUnits; ++u) {
    const int i = (int)threadIdx.x + u * kRepackThreads, c = i % kW, w = i / kW;
    nibble_transpose8(R[u]);
    const int bl = c >> 3;
#pragma unroll
    for (int col = 0; col < 8; ++col) {
      const int r = 8 * (c & 7) + col;
      out[bl][r][w ^ out_swizzle(bl, r)] = R[u][awq_slot_of_col(col)];
    }
  }
  __syncthreads();

  for (int bl = 0; bl < kRepackBlocks; ++bl) {
    const int b = bfirst + bl;
    if (b >= b1) break;
    uint8_t *chunk = packed + kHeaderBytes + ((size_t)b * KT + t) * CB;
    // the 4 KB of codes in layout order, a warp storing 128 contiguous bytes at a time
    uint32_t *codes = reinterpret_cast<uint32_t *>(chunk);
#pragma unroll
    for (int u = 0; u < kBlockN * 16 / kRepackThreads; ++u) {
      const int i = (int)threadIdx.x + u * kRepackThreads;
      if (in_extent(codes + i, 4, packed, pext, err)) codes[i] = out[bl][i >> 4][(i & 15) ^ out_swizzle(bl, i >> 4)];
    }

    // Meta: per group of the chunk, 64 scales and 64 zero nibbles in lane order.  Layout group
    // grp covers rows [grp g, grp g + g); its scales and zeros are row (grp g) / gsrc of the
    // source tensors (gsrc == g, or gsrc == K for one group over all of K).
    for (int i = threadIdx.x; i < gpc * kBlockN; i += blockDim.x) {
      const int l = i / kBlockN, r = i % kBlockN;  // source column 64b + r
      uint16_t *dst = reinterpret_cast<uint16_t *>(chunk + kCodeBytes + l * kGroupMetaBytes) + meta_pos(r);
      if (in_extent(dst, 2, packed, pext, err)) *dst = sin[bl][l][r];
    }
    if (threadIdx.x < gpc * 8) {
      const int l = threadIdx.x >> 3, wi = threadIdx.x & 7;
      uint32_t o = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int r = meta_row(8 * wi + j);
        o |= ((zin[l][8 * bl + (r >> 3)] >> (4 * awq_slot_of_col(r & 7))) & 0xFu) << (4 * j);
      }
      uint32_t *dst = reinterpret_cast<uint32_t *>(chunk + kCodeBytes + l * kGroupMetaBytes + kScaleBytes) + wi;
      if (in_extent(dst, 4, packed, pext, err)) *dst = o;
    }
  }
}

}  // namespace

cudaError_t launch_repack(const int32_t *qweight, int64_t ldq, const int32_t *qzeros, int64_t ldz,
                          const uint16_t *scales, int64_t lds, int K, int N, int g, int gsrc, int dtype,
                          int n0, int n1, void *packed, int *err, cudaStream_t stream) {
  int b0 = n0 / kBlockN;
  int b1 = (n1 + kBlockN - 1) / kBlockN;
  int KT = num_ktiles(K);
  dim3 grid((b1 - b0 + kRepackBlocks - 1) / kRepackBlocks, KT);
  repack_kernel<<<grid, kRepackThreads, 0, stream>>>(qweight, ldq, qzeros, ldz, scales, lds, K, N, g, gsrc, dtype, n0, n1,
                                          b0, b1, KT, static_cast<uint8_t *>(packed), err);
  return cudaGetLastError();
}

}  // namespace w4a16
