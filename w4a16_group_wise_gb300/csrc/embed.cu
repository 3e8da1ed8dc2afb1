// embed.cu -- gather of the quantized tied embedding: out[t][k] = W[k][ids[t]], bit-exact, in the
// layer's element type (fp16 or bf16).
//
// The LM head's packed weight doubles as the embedding table: the head is tied to the
// embedding (vllm-omni commit "cpu_int4: repack weights in n-blocks, to bound the load-time
// peak": "embedding 131072 x 2048 ... tied, so it is also the head"; commit "Add cpu_int4 ...":
// "the quantized tied embedding").  A token id n selects column n of W [K][N], and its
// embedding row is that column dequantized: fp16((q[k][n] - z[k/g][n]) * s[k/g][n]) with the
// same single rounding as the dequantized weight (dq.cuh).
//
// In the packed layout a column is one 64-byte row of each of its n-block's chunks, so a token
// reads K/2 bytes of codes in 64-byte runs plus its scale and zero per group.  One CTA of 128
// threads takes a token and 8 chunks (1024 k): thread i converts code word i % 16 (8 k) of
// chunk i / 16 and stores 16 bytes of the output row, so a warp's stores are 512 contiguous
// bytes.  An id outside [0, N) gives a row of zeros and records a device-side error.
#include <cuda_runtime.h>

#include "bounds.cuh"
#include "dq.cuh"
#include "kernels.h"
#include "layout.cuh"

namespace w4a16 {
namespace {

constexpr int kEmbedThreads = 128;
constexpr int kChunksPerCta = kEmbedThreads / 16;

template <class T>
__global__ void __launch_bounds__(kEmbedThreads) embed_kernel(const int32_t *__restrict__ ids,
                                                              const uint8_t *__restrict__ packed, int K, int N,
                                                              int g, int KT, uint16_t *__restrict__ out, int *err) {
  const int t = blockIdx.x;
  const int c = blockIdx.y * kChunksPerCta + threadIdx.x / 16;  // chunk (k-tile) of this thread
  const int w = threadIdx.x % 16;                                // code word of the column row
  const int k0 = c * kTileK + 8 * w;
  const int ntok = gridDim.x;  // tokens: one CTA row per id
  const long long pext = packed_extent(K, N, g), oext = 2LL * ntok * K;
  const Header *h = reinterpret_cast<const Header *>(packed);
  const bool hdr_ok = in_extent(h, sizeof(Header), packed, pext, err) && h->magic == kMagic && h->version == kLayoutVersion && h->K == K && h->N == N && h->g == g &&
                      h->dtype == T::kDtype;
  if (!hdr_ok) {
    if (threadIdx.x == 0 && blockIdx.y == 0) atomicOr(err, 1);
    return;  // a mismatched buffer writes nothing
  }
  if (c >= KT || k0 >= K) return;
  const int n = in_extent(ids + t, 4, ids, 4LL * ntok, err) ? __ldg(ids + t) : 0;
  uint4 o = make_uint4(0, 0, 0, 0);
  if (n < 0 || n >= N) {
    if (threadIdx.x == 0 && blockIdx.y == 0) atomicOr(err, 4);
  } else {
    const int b = n / kBlockN, rr = n % kBlockN, p = meta_pos(rr);
    const uint8_t *chunk = packed + kHeaderBytes + ((size_t)b * KT + c) * chunk_bytes(g);
    const uint32_t *wp = reinterpret_cast<const uint32_t *>(chunk + rr * kRowBytes) + w;
    const uint8_t *meta = chunk + kCodeBytes + ((8 * w) / g) * kGroupMetaBytes;
    const uint16_t *sp = reinterpret_cast<const uint16_t *>(meta) + p;
    const uint32_t *zp = reinterpret_cast<const uint32_t *>(meta + kScaleBytes) + p / 8;
    const uint32_t word = in_extent(wp, 4, packed, pext, err) ? __ldg(wp) : 0u;
    const uint32_t s = in_extent(sp, 2, packed, pext, err) ? __ldg(sp) : 0u;
    const uint32_t zw = in_extent(zp, 4, packed, pext, err) ? __ldg(zp) : 0u;
    uint32_t v[4];
    T::qz(word, T::zb((zw >> (4 * (p % 8))) & 0xFu), v);
    const uint32_t s2 = s * 0x00010001u;
    o = make_uint4(T::mul2(v[0], s2), T::mul2(v[1], s2), T::mul2(v[2], s2), T::mul2(v[3], s2));
  }
  if (in_extent(out + (size_t)t * K + k0, 16, out, oext, err)) *reinterpret_cast<uint4 *>(out + (size_t)t * K + k0) = o;
}

}  // namespace

cudaError_t launch_embed(const int32_t *ids, int T, const void *packed, int K, int N, int g, int dtype,
                         uint16_t *out, int *err, cudaStream_t stream) {
  const int KT = num_ktiles(K);
  dim3 grid(T, (KT + kChunksPerCta - 1) / kChunksPerCta);
  const uint8_t *p = static_cast<const uint8_t *>(packed);
  if (dtype == kDtypeBf16)
    embed_kernel<Bf16><<<grid, kEmbedThreads, 0, stream>>>(ids, p, K, N, g, KT, out, err);
  else
    embed_kernel<Fp16><<<grid, kEmbedThreads, 0, stream>>>(ids, p, K, N, g, KT, out, err);
  return cudaGetLastError();
}

}  // namespace w4a16
