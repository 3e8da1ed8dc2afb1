// dequant.cu -- packed layout -> W[K][N] in the layer's element type (fp16 or bf16), bit-exact.
//
// The analogue of _dequantize_from_int4pack (vllm-omni commit "cpu_int4: dequantize prefill
// weights from the tinygemm layout, not a copy"): decoding the packed layout is a
// de-interleave, and the result must be bit-exact against the straightforward dequantizer,
// including an N that does not tile the 64-column block (N = 80).  Every weight is
// fp16((q - z) * s), or bf16((q - z) * s) for a bf16 layer, with one rounding (see dq.cuh).
//
// One CTA per chunk (64 columns x 128 rows of K): 256 (column-row, 32-k span) units are
// converted into a shared [128 k][64 n] tile, then written out as 16-byte row segments.
#include <cuda_runtime.h>

#include "bounds.cuh"
#include "dq.cuh"
#include "kernels.h"
#include "layout.cuh"

namespace w4a16 {
namespace {

constexpr int kTileLd = kBlockN + 8;  // padded row of the shared tile (halves), 144 bytes

template <class T>
__global__ void __launch_bounds__(128) dequant_kernel(const uint8_t *__restrict__ packed, int K, int N,
                                                      int g, int KT, uint16_t *__restrict__ W, int *err) {
  __shared__ __align__(16) uint16_t tile[kTileK][kTileLd];
  __shared__ int bad;
  const int b = blockIdx.x, t = blockIdx.y;
  const int CB = chunk_bytes(g);
  const uint8_t *chunk = packed + kHeaderBytes + ((size_t)b * KT + t) * CB;
  const long long pext = packed_extent(K, N, g), wext = 2LL * K * N;

  if (threadIdx.x == 0) {
    const Header *h = reinterpret_cast<const Header *>(packed);
    bad = (!in_extent(h, sizeof(Header), packed, pext, err) || h->magic != kMagic || h->version != kLayoutVersion || h->K != K || h->N != N || h->g != g ||
           h->dtype != T::kDtype);
    if (bad) atomicOr(err, 1);
  }

  for (int u = threadIdx.x; u < kBlockN * 4; u += blockDim.x) {
    const int r = u % kBlockN, span = u / kBlockN;  // column-row, 32-k span
    const uint8_t *cp = chunk + r * kRowBytes + span * 16;
    uint4 c = in_extent(cp, 16, packed, pext, err) ? __ldg(reinterpret_cast<const uint4 *>(cp)) : make_uint4(0, 0, 0, 0);
    const uint8_t *meta = chunk + kCodeBytes + ((32 * span) / g) * kGroupMetaBytes;
    const int p = meta_pos(r);
    const uint16_t *sp = reinterpret_cast<const uint16_t *>(meta) + p;
    const uint32_t *zp = reinterpret_cast<const uint32_t *>(meta + kScaleBytes) + p / 8;
    uint32_t s = in_extent(sp, 2, packed, pext, err) ? __ldg(sp) : 0u;
    uint32_t zw = in_extent(zp, 4, packed, pext, err) ? __ldg(zp) : 0u;
    ZeroBias zb = T::zb((zw >> (4 * (p % 8))) & 0xFu);
    uint32_t s2 = s * 0x00010001u;
    uint32_t words[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      uint32_t v[4];
      T::qz(words[w], zb, v);
      const int k0 = 32 * span + 8 * w;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        uint32_t wv = T::mul2(v[e], s2);
        tile[k0 + 2 * e][r] = (uint16_t)(wv & 0xFFFFu);
        tile[k0 + 2 * e + 1][r] = (uint16_t)(wv >> 16);
      }
    }
  }
  __syncthreads();
  if (bad) return;

  const int kb = t * kTileK;
  for (int i = threadIdx.x; i < kTileK * (kBlockN / 8); i += blockDim.x) {
    const int kk = i / (kBlockN / 8), v = i % (kBlockN / 8);
    const int k = kb + kk, n = b * kBlockN + 8 * v;
    if (k < K && n < N && in_extent(W + (size_t)k * N + n, 16, W, wext, err))
      *reinterpret_cast<uint4 *>(W + (size_t)k * N + n) = *reinterpret_cast<const uint4 *>(&tile[kk][8 * v]);
  }
}

}  // namespace

cudaError_t launch_dequant(const void *packed, int K, int N, int g, int dtype, uint16_t *W, int *err,
                           cudaStream_t stream) {
  int KT = num_ktiles(K);
  dim3 grid(num_nblocks(N), KT);
  const uint8_t *p = static_cast<const uint8_t *>(packed);
  if (dtype == kDtypeBf16)
    dequant_kernel<Bf16><<<grid, 128, 0, stream>>>(p, K, N, g, KT, W, err);
  else
    dequant_kernel<Fp16><<<grid, 128, 0, stream>>>(p, K, N, g, KT, W, err);
  return cudaGetLastError();
}

}  // namespace w4a16
