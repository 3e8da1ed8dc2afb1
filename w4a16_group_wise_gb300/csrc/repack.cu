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
// size).  One CTA writes one self-contained chunk, so any n-range can be repacked on its own.
#include <cuda_runtime.h>

#include "kernels.h"
#include "layout.cuh"

namespace w4a16 {
namespace {

// column offset inside an AWQ word -> its nibble slot (inverse of {0,2,4,6,1,3,5,7})
__device__ __forceinline__ int awq_slot_of_col(int c) { return (c & 1) ? 4 + (c >> 1) : (c >> 1); }

// lane-order position p -> column-row r (inverse of meta_pos)
__device__ __forceinline__ int meta_row(int p) { return 16 * ((p % 8) / 2) + 8 * (p % 2) + p / 8; }

__global__ void __launch_bounds__(256) repack_kernel(
    const int32_t *__restrict__ qweight, int64_t ldq, const int32_t *__restrict__ qzeros,
    int64_t ldz, const uint16_t *__restrict__ scales, int64_t lds, int K, int N, int g, int gsrc, int dtype,
    int n0, int b0, int KT, uint8_t *__restrict__ packed) {
  const int b = b0 + blockIdx.x;  // n-block
  const int t = blockIdx.y;       // k-tile
  const int kb = t * kTileK;
  const int CB = chunk_bytes(g);
  uint8_t *chunk = packed + kHeaderBytes + ((size_t)b * KT + t) * CB;

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
    reinterpret_cast<uint32_t *>(packed)[threadIdx.x] = v;
  }

  // Stage the 128 x 8 AWQ words of this chunk (rows past K and columns past N read as 0).
  __shared__ uint32_t in[kTileK][8];
  for (int i = threadIdx.x; i < kTileK * 8; i += blockDim.x) {
    int kk = i >> 3, c = i & 7;
    int k = kb + kk, n = b * kBlockN + 8 * c;
    uint32_t w = 0;
    if (k < K && n < N) w = (uint32_t)qweight[(int64_t)k * ldq + (n - n0) / 8];
    in[kk][c] = w;
  }
  __syncthreads();

  // Codes: row r (column 64b + r), word w covers k = kb + 8w + slot_k(j) in slot j.
  uint32_t *codes = reinterpret_cast<uint32_t *>(chunk);
  for (int i = threadIdx.x; i < kBlockN * 16; i += blockDim.x) {
    int r = i >> 4, w = i & 15;
    int c = r >> 3, in_slot = awq_slot_of_col(r & 7);
    uint32_t out = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      uint32_t code = (in[8 * w + slot_k(j)][c] >> (4 * in_slot)) & 0xFu;
      out |= code << (4 * j);
    }
    codes[i] = out;
  }

  // Meta: per group of the chunk, 64 scales and 64 zero nibbles in lane order.  Layout group
  // grp covers rows [grp g, grp g + g); its scales and zeros are row (grp g) / gsrc of the
  // source tensors (gsrc == g, or gsrc == K for one group over all of K).
  const int gpc = kTileK / g;  // groups per chunk
  const int G = K / g;
  for (int i = threadIdx.x; i < gpc * kBlockN; i += blockDim.x) {
    int l = i / kBlockN, p = i % kBlockN;
    int grp = t * gpc + l, n = b * kBlockN + meta_row(p);
    int sg = (grp * g) / gsrc;
    uint16_t s = 0;
    if (grp < G && n < N) s = scales[(int64_t)sg * lds + (n - n0)];
    reinterpret_cast<uint16_t *>(chunk + kCodeBytes + l * kGroupMetaBytes)[p] = s;
  }
  for (int i = threadIdx.x; i < gpc * 8; i += blockDim.x) {
    int l = i / 8, wi = i % 8;
    int grp = t * gpc + l;
    int sg = (grp * g) / gsrc;
    uint32_t out = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      int n = b * kBlockN + meta_row(8 * wi + j);
      uint32_t z = 0;
      if (grp < G && n < N) {
        uint32_t zw = (uint32_t)qzeros[(int64_t)sg * ldz + (n - n0) / 8];
        z = (zw >> (4 * awq_slot_of_col(n & 7))) & 0xFu;
      }
      out |= z << (4 * j);
    }
    reinterpret_cast<uint32_t *>(chunk + kCodeBytes + l * kGroupMetaBytes + kScaleBytes)[wi] = out;
  }
}

}  // namespace

cudaError_t launch_repack(const int32_t *qweight, int64_t ldq, const int32_t *qzeros, int64_t ldz,
                          const uint16_t *scales, int64_t lds, int K, int N, int g, int gsrc, int dtype,
                          int n0, int n1, void *packed, cudaStream_t stream) {
  int b0 = n0 / kBlockN;
  int b1 = (n1 + kBlockN - 1) / kBlockN;
  int KT = num_ktiles(K);
  dim3 grid(b1 - b0, KT);
  repack_kernel<<<grid, 256, 0, stream>>>(qweight, ldq, qzeros, ldz, scales, lds, K, N, g, gsrc, dtype, n0,
                                          b0, KT, static_cast<uint8_t *>(packed));
  return cudaGetLastError();
}

}  // namespace w4a16
