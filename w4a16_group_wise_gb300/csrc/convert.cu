// convert.cu -- AWQ packing -> the GPTQ-style "standard" packing, integer-exact.
//
// vLLM walkthrough "Carga de capas cuantizadas: AWQ / GPTQ / Marlin / fp8", section
// "Motivacion de diseno": AWQ packs its codes along the output dimension in a non-standard
// order, where the standard (GPTQ-style) checkpoints pack along the input dimension in plain
// order.  Out:
//   qweight_std int32 [K/8][N]:   nibble slot j (bits 4j..4j+3) of word (r, n) = q[8r + j][n];
//   qzeros_std  int32 [K/g][N/8]: nibble slot j of word (G, c) = z[G][8c + j];
// the scales are the same tensor in both formats.  In AWQ words column 8c + o sits in slot
// {0,4,1,5,2,6,3,7}[o] (the inverse of the slot order {0,2,4,6,1,3,5,7}).
//
// qweight: one thread per (row octet, AWQ word column) reads the 8 words of rows 8r..8r+7
// (consecutive threads read consecutive words), transposes their 8 x 8 nibbles in registers and
// writes the 8 output words of its column octet as 32 contiguous bytes.  qzeros: one thread per
// word permutes its nibbles, in CTAs appended to the same grid (one launch for both tensors).
#include <cuda_runtime.h>

#include "bounds.cuh"
#include "kernels.h"
#include "nibble.cuh"

namespace w4a16 {
namespace {

__device__ __forceinline__ int awq_slot(int o) { return (o & 1) ? 4 + (o >> 1) : (o >> 1); }

constexpr int kConvertThreads = 256;

// CTAs [0, qblocks) convert qweight, the rest qzeros.
__global__ void __launch_bounds__(kConvertThreads) awq_to_standard_kernel(
    const int32_t *__restrict__ qa, const int32_t *__restrict__ za, int K, int N, int64_t zwords,
    unsigned qblocks, int32_t *__restrict__ qs, int32_t *__restrict__ zs, int *err) {
  if (blockIdx.x >= qblocks) {  // one zero word per thread
    const int64_t i = (int64_t)(blockIdx.x - qblocks) * kConvertThreads + threadIdx.x;
    if (i >= zwords) return;
    if (!in_extent(za + i, 4, za, 4 * zwords, err) || !in_extent(zs + i, 4, zs, 4 * zwords, err)) return;
    const uint32_t src = (uint32_t)__ldg(za + i);
    uint32_t w = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) w |= ((src >> (4 * awq_slot(j))) & 0xFu) << (4 * j);
    zs[i] = (int32_t)w;
    return;
  }
  const long long ext = 4LL * (K / 8) * N;  // both tensors: K*N/8 words
  const int C = N / 8;
  const int64_t i = (int64_t)blockIdx.x * kConvertThreads + threadIdx.x;  // (row octet r, word column c)
  if (i >= (int64_t)(K / 8) * C) return;
  const int r = (int)(i / C), c = (int)(i % C);
  uint32_t R[8];  // row 8r + j; after the transpose R[p] holds nibble p of rows 8r .. 8r+7
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int32_t *src = qa + (int64_t)(8 * r + j) * C + c;
    R[j] = in_extent(src, 4, qa, ext, err) ? (uint32_t)__ldg(src) : 0u;
  }
  nibble_transpose8(R);
  uint4 *dst = reinterpret_cast<uint4 *>(qs + (int64_t)r * N + 8 * c);  // 32 contiguous bytes
  if (!in_extent(dst, 32, qs, ext, err)) return;
  // column 8c + o: AWQ slot awq_slot(o)
  dst[0] = make_uint4(R[awq_slot(0)], R[awq_slot(1)], R[awq_slot(2)], R[awq_slot(3)]);
  dst[1] = make_uint4(R[awq_slot(4)], R[awq_slot(5)], R[awq_slot(6)], R[awq_slot(7)]);
}

}  // namespace

cudaError_t launch_awq_to_standard(const int32_t *qweight_awq, const int32_t *qzeros_awq, int K, int N,
                                   int zero_rows, int32_t *qweight_std, int32_t *qzeros_std, int *err,
                                   cudaStream_t stream) {
  const int64_t qthreads = (int64_t)(K / 8) * (N / 8), zwords = (int64_t)zero_rows * (N / 8);
  const unsigned qblocks = (unsigned)((qthreads + kConvertThreads - 1) / kConvertThreads);
  const unsigned zblocks = (unsigned)((zwords + kConvertThreads - 1) / kConvertThreads);
  if (qblocks + zblocks == 0) return cudaSuccess;
  awq_to_standard_kernel<<<qblocks + zblocks, kConvertThreads, 0, stream>>>(qweight_awq, qzeros_awq, K, N, zwords,
                                                                            qblocks, qweight_std, qzeros_std, err);
  return cudaGetLastError();
}

}  // namespace w4a16
