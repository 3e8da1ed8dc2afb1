// gemv.cu -- decode path of y = x . W for few rows of x (M <= 16 per m-block).
//
// Why a separate path: "single-stream decode reads every weight to emit one token, so bits
// per weight set the token rate" (vllm-omni commit "Add cpu_int4, an asymmetric 4-bit weight
// path for vLLM's CPU backend").  The kernel streams the packed weights exactly once with
// 128-bit coalesced loads, converts nibbles to fp16 in registers (dq.cuh), and lets the tensor
// pipe do the multiply-adds (mma.sync m16n8k16, fp16 x fp16 -> fp32) so that the conversion
// work, not the FMAs, is what the CUDA cores issue.  The weight tile is the A operand
// (16 columns n x 16 k) and x^T the B operand (16 k x 8 rows m), so M <= 8 costs one MMA per
// 256 weights and M <= 16 two.
//
// k permutation: inside a 128-k chunk, lane (r8 = lane/4, t = lane%4) owns the 32-k span
// [32t, 32t+32) of its column-rows.  MMA step j (0..7) maps the fragment's logical k
// {2t, 2t+1, 2t+8, 2t+9} to physical k 32t + 4j + {0, 1, 2, 3}; A and B fragments use the same
// map (both index k by t), so the products are unchanged and every lane reads contiguous data.
//
// Scale: for g = 128 a chunk is one group, so the MMA chain over the chunk's 8 steps sums
// (q - z) * x exactly in fp32 and the fp32 scale is applied once per (column, row of x)
// afterwards.  For g = 32 / 64 the chain spans several groups and each weight is multiplied by
// its scale in fp16 (the exact fp16 weight) before the MMA.
//
// Split of K: the W warps of a CTA take the CTA's chunks round-robin; the S CTAs of a thread
// block cluster (S <= 8) take consecutive K ranges of the same n-block.  Partial sums are added
// in a fixed order (warps 0..W-1, then cluster ranks 0..S-1 read through distributed shared
// memory), so y is bit-identical from run to run and no global workspace is needed.
#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include "dq.cuh"
#include "kernels.h"
#include "layout.cuh"

namespace cg = cooperative_groups;

namespace w4a16 {
namespace {

constexpr int kMaxWarps = 4;
constexpr int kMaxCluster = 8;

__device__ __forceinline__ uint4 ld_stream(const void *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void mma16816(float d[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// MB: 8-row blocks of x handled per CTA (1: M <= 8, 2: M <= 16).  FACTOR: scale applied per
// chunk in fp32 (g == 128) instead of per weight in fp16.
template <int MB, bool FACTOR>
__global__ void __launch_bounds__(kMaxWarps * 32) gemv_kernel(
    const uint16_t *__restrict__ x, const uint8_t *__restrict__ packed, int M, int N, int K, int g,
    int KT, int chunks_per_cta, uint16_t *__restrict__ y, int *err) {
  constexpr int kVals = 16 * MB;  // accumulator values per lane: 4 row-tiles x MB x 4
  __shared__ float red[kMaxWarps][kVals][32];
  __shared__ float part[kVals * 32];
  __shared__ int bad;

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const int r8 = lane >> 2, t = lane & 3;
  const int b = blockIdx.x;
  const int S = gridDim.y, s = blockIdx.y;
  const int m0 = blockIdx.z * 8 * MB;
  const int CB = chunk_bytes(g);
  const int kt_begin = s * chunks_per_cta;
  const int kt_end = min(KT, kt_begin + chunks_per_cta);
  const uint8_t *body = packed + kHeaderBytes + (size_t)b * KT * CB;

  float acc[4][MB][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int mb = 0; mb < MB; ++mb)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[i][mb][c] = 0.f;

#pragma unroll 1
  for (int kt = kt_begin + warp; kt < kt_end; kt += nwarps) {
    const uint8_t *chunk = body + (size_t)kt * CB;
    uint4 cw[4][2];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int h = 0; h < 2; ++h) cw[i][h] = ld_stream(chunk + (16 * i + r8 + 8 * h) * kRowBytes + 16 * t);
    const uint8_t *meta = chunk + kCodeBytes + ((32 * t) / g) * kGroupMetaBytes;
    const uint4 sc = __ldg(reinterpret_cast<const uint4 *>(meta) + r8);
    const uint32_t zw = __ldg(reinterpret_cast<const uint32_t *>(meta + kScaleBytes) + r8);

    const int kx = kt * kTileK + 32 * t;
    uint4 xf[MB][4];
#pragma unroll
    for (int mb = 0; mb < MB; ++mb) {
      const int m = m0 + 8 * mb + r8;
      const bool ok = (m < M) && (kx < K);
      const uint4 *xp = reinterpret_cast<const uint4 *>(x + (size_t)(ok ? m : 0) * K + (ok ? kx : 0));
#pragma unroll
      for (int q = 0; q < 4; ++q) xf[mb][q] = ok ? __ldg(xp + q) : make_uint4(0, 0, 0, 0);
    }
    const uint32_t scw[4] = {sc.x, sc.y, sc.z, sc.w};

#pragma unroll
    for (int i = 0; i < 4; ++i) {
      // scales of rows 16i + r8 (h = 0) and 16i + r8 + 8 (h = 1): halves 2i and 2i+1 of sc
      const uint32_t s_lo = scw[i] & 0xFFFFu, s_hi = scw[i] >> 16;
      const ZeroBias zb0 = zero_bias((zw >> (8 * i)) & 0xFu);
      const ZeroBias zb1 = zero_bias((zw >> (8 * i + 4)) & 0xFu);
      float d[MB][4];
#pragma unroll
      for (int mb = 0; mb < MB; ++mb)
#pragma unroll
        for (int c = 0; c < 4; ++c) d[mb][c] = 0.f;
      const uint32_t w0[4] = {cw[i][0].x, cw[i][0].y, cw[i][0].z, cw[i][0].w};
      const uint32_t w1[4] = {cw[i][1].x, cw[i][1].y, cw[i][1].z, cw[i][1].w};
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        uint32_t v0[4], v1[4];
        word_to_qz(w0[w], zb0, v0);
        word_to_qz(w1[w], zb1, v1);
        if (!FACTOR) {
          const uint32_t s20 = s_lo * 0x00010001u, s21 = s_hi * 0x00010001u;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            v0[e] = hmul2_u32(v0[e], s20);
            v1[e] = hmul2_u32(v1[e], s21);
          }
        }
#pragma unroll
        for (int mb = 0; mb < MB; ++mb) {
          float *dst = FACTOR ? d[mb] : acc[i][mb];
          const uint32_t xs[4] = {xf[mb][w].x, xf[mb][w].y, xf[mb][w].z, xf[mb][w].w};
          mma16816(dst, v0[0], v1[0], v0[1], v1[1], xs[0], xs[1]);  // k 8w + 0..3
          mma16816(dst, v0[2], v1[2], v0[3], v1[3], xs[2], xs[3]);  // k 8w + 4..7
        }
      }
      if (FACTOR) {
        const float f0 = __half2float(__ushort_as_half((unsigned short)s_lo));
        const float f1 = __half2float(__ushort_as_half((unsigned short)s_hi));
#pragma unroll
        for (int mb = 0; mb < MB; ++mb) {
          acc[i][mb][0] = fmaf(f0, d[mb][0], acc[i][mb][0]);
          acc[i][mb][1] = fmaf(f0, d[mb][1], acc[i][mb][1]);
          acc[i][mb][2] = fmaf(f1, d[mb][2], acc[i][mb][2]);
          acc[i][mb][3] = fmaf(f1, d[mb][3], acc[i][mb][3]);
        }
      }
    }
  }

  // ---- deterministic reduction: warps in order, then cluster ranks in order
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int mb = 0; mb < MB; ++mb)
#pragma unroll
      for (int c = 0; c < 4; ++c) red[warp][(i * MB + mb) * 4 + c][lane] = acc[i][mb][c];
  if (threadIdx.x == 0) {
    const Header *h = reinterpret_cast<const Header *>(packed);
    bad = (h->magic != kMagic || h->version != kLayoutVersion || h->K != K || h->N != N || h->g != g);
    if (bad && b == 0 && s == 0 && blockIdx.z == 0) atomicExch(err, 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < kVals * 32; e += blockDim.x) {
    float v = 0.f;
    for (int w = 0; w < nwarps; ++w) v += red[w][e / 32][e % 32];
    part[e] = v;
  }

  bool write = true;
  if (S > 1) {
    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();
    write = cluster.block_rank() == 0;
    if (write) {
      for (int e = threadIdx.x; e < kVals * 32; e += blockDim.x) {
        float v = 0.f;
        for (int rk = 0; rk < S; ++rk) v += cluster.map_shared_rank(part, rk)[e];
        part[e] = v;  // only rank 0 rewrites its own entry after every rank has been read
      }
    }
    cluster.sync();
  } else {
    __syncthreads();
  }
  if (!write || bad) return;
  if (S > 1) __syncthreads();

  for (int e = threadIdx.x; e < kVals * 32; e += blockDim.x) {
    const int ln = e % 32, vi = e / 32;
    const int c = vi % 4, mb = (vi / 4) % MB, i = vi / (4 * MB);
    const int row = 16 * i + (ln >> 2) + 8 * (c >> 1);
    const int m = m0 + 8 * mb + 2 * (ln & 3) + (c & 1);
    const int n = b * kBlockN + row;
    if (m < M && n < N) y[(size_t)m * N + n] = __half_as_ushort(__float2half_rn(part[e]));
  }
}

template <int MB, bool FACTOR>
cudaError_t launch_variant(dim3 grid, int warps, int S, const uint16_t *x, const uint8_t *packed, int M,
                           int N, int K, int g, int KT, int cpc, uint16_t *y, int *err,
                           cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(32 * warps);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  int na = 0;
  if (S > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = 1;
    attr[na].val.clusterDim.y = S;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, gemv_kernel<MB, FACTOR>, x, packed, M, N, K, g, KT, cpc, y, err);
}

int sm_count() {
  static int count = 0;
  if (!count) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&count, cudaDevAttrMultiProcessorCount, dev);
    if (count <= 0) count = 148;
  }
  return count;
}

}  // namespace

cudaError_t launch_gemv(const uint16_t *x, const void *packed, int M, int N, int K, int g, uint16_t *y,
                        int *err, cudaStream_t stream) {
  const int NB = num_nblocks(N), KT = num_ktiles(K);
  const int MB = (M <= 8) ? 1 : 2;
  const int mblocks = (M + 8 * MB - 1) / (8 * MB);
  // Split K over a cluster until the grid covers the GPU about twice.
  int S = 1;
  while (S < kMaxCluster && S * 2 <= KT && (long)NB * S * mblocks < 2L * sm_count()) S *= 2;
  const int cpc = (KT + S - 1) / S;  // chunks per CTA
  const int warps = cpc < kMaxWarps ? cpc : kMaxWarps;
  dim3 grid(NB, S, mblocks);
  const uint8_t *p = static_cast<const uint8_t *>(packed);
  const bool factor = (g == kTileK);
  if (MB == 1)
    return factor ? launch_variant<1, true>(grid, warps, S, x, p, M, N, K, g, KT, cpc, y, err, stream)
                  : launch_variant<1, false>(grid, warps, S, x, p, M, N, K, g, KT, cpc, y, err, stream);
  return factor ? launch_variant<2, true>(grid, warps, S, x, p, M, N, K, g, KT, cpc, y, err, stream)
                : launch_variant<2, false>(grid, warps, S, x, p, M, N, K, g, KT, cpc, y, err, stream);
}

}  // namespace w4a16
