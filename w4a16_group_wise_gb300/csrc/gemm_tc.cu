// gemm_tc.cu -- tensor-core path of y = x . W for many rows of x (prefill).
//
// Why a second path: the CPU plugin found that a kernel which dequantizes once per row of
// activations is linear in the batch (12.9x slower than bf16 at 512 rows), so wide batches
// unpack the weight once and run an ordinary dense GEMM (vllm-omni commit "Add cpu_int4, an
// asymmetric 4-bit weight path for vLLM's CPU backend").  Here the unpacking is fused into the
// GEMM: each 128 x 128 weight tile is dequantized once per CTA into shared memory and consumed
// by the 5th-generation tensor cores (tcgen05.mma, fp16 x fp16 -> fp32 in tensor memory); no
// dequantized W ever reaches HBM.
//
// Orientation: D[n][m] = sum_k W^T[n][k] * x^T[k][m], i.e. the MMA's M dimension (128) runs
// over output columns n and its N dimension (BM <= 256) over rows m of x, so few rows of x
// waste no tensor work.  Per k-block of 128 (one packed chunk):
//  - one lane of warp 0 loads the x tile (BM rows x 128 k, fp16) with two TMA copies into a
//    128-byte-swizzled K-major tile (rows past M and k past K read as 0);
//  - warps 4..7 (one thread per column-row) load that row's 64 code bytes and its scales and
//    zeros, convert them to the exact fp16 weights fp16((q - z) * s) (dq.cuh) and store them into
//    the A tile with the same 128-byte swizzle, then fence the writes to the async proxy;
//  - one lane of warp 1 issues 8 MMAs (K = 16 each) once both operands are in place and
//    commits them to the stage's "empty" barrier, which frees the stage when they complete.
// The stages form a ring; after the last k-block the accumulator is committed to a barrier,
// and all 8 warps read it back (tcgen05.ld, 32 lanes x 16 columns each), round to fp16 and
// store y.  Every wait is bounded: on a timeout the kernel records an error, drains, frees
// tensor memory and skips the store.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "dq.cuh"
#include "kernels.h"
#include "layout.cuh"
#include "ptx.cuh"

namespace w4a16 {
namespace {

constexpr int kBN = 128;          // weight rows (output columns n) per CTA = MMA M
constexpr int kBK = 128;          // k per stage (one packed chunk)
constexpr int kAtomK = 64;        // k per 128-byte swizzle atom (fp16)
constexpr int kAStageBytes = kBN * kBK * 2;  // 32 KB
constexpr int kMaxStages = 4;
constexpr int kThreads = 256;

struct GemmSmem {
  int stages, bm;
  int a_off, b_off, stage_bytes, total;
};

__host__ __device__ inline GemmSmem gemm_smem(int bm, int stages) {
  GemmSmem s;
  s.bm = bm;
  s.stages = stages;
  s.stage_bytes = kAStageBytes + bm * kBK * 2;
  s.a_off = 0;
  s.b_off = kAStageBytes;
  s.total = stages * s.stage_bytes;
  return s;
}

// --------------------------------------------------------------------------- tcgen05 wrappers

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t sw128_desc(const void *p) {
  const uint64_t addr = smem_u32(p);
  return ((addr >> 4) & 0x3FFFull) | (1ull << 16) | (64ull << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor, kind::f16: fp16 A and B (K-major), fp32 D, M = 128, N = n.
__host__ __device__ inline uint32_t idesc_f16(int n) {
  return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}

__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 32 lanes x 16 consecutive 32-bit columns (one lane per thread of the warp).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int c0, int c1, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(map), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}

// --------------------------------------------------------------------------- the kernel

__global__ void __launch_bounds__(kThreads, 1) gemm_tc_kernel(const __grid_constant__ CUtensorMap xmap,
                                                               const uint8_t *__restrict__ packed, int M, int N,
                                                               int K, int g, int KT, int bm, int stages,
                                                               int tmem_cols, uint16_t *__restrict__ y, int *err) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte alignment of the operand tiles (the swizzle pattern repeats every 1024 bytes)
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t full_bar[kMaxStages], empty_bar[kMaxStages], accum_bar;
  __shared__ uint32_t tmem_base;
  __shared__ int flags;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const GemmSmem L = gemm_smem(bm, stages);
  const int n0 = blockIdx.x * kBN, m0 = blockIdx.y * bm;
  const int NB = num_nblocks(N);
  const int CB = chunk_bytes(g);
  const uint32_t x_bytes = (uint32_t)bm * kBK * 2;

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full_bar[s], 1 + 128);  // TMA expect-tx arrival + 128 dequant threads
      mbar_init(&empty_bar[s], 1);       // one tcgen05.commit per use
    }
    mbar_init(&accum_bar, 1);
    flags = 0;
    fence_mbar_init();
  }
  if (warp == 1) {  // the whole warp allocates tensor memory: tmem_cols fp32 columns x 128 lanes
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_base)),
                 "r"(tmem_cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;
  griddep_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------ x tiles by TMA (one lane)
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(&xmap) : "memory");
      griddep_wait();  // x may be the previous kernel's output
      bool ok = true;
      int issued = 0;
      for (int kb = 0; kb < KT; ++kb) {
        const int s = kb % stages, use = kb / stages;
        if (use > 0 && !(ok = mbar_wait_bounded(&empty_bar[s], (use - 1) & 1))) break;
        uint8_t *b = smem + s * L.stage_bytes + L.b_off;
        mbar_arrive_expect_tx(&full_bar[s], x_bytes);
        tma_load_2d(b, &xmap, kb * kBK, m0, &full_bar[s]);
        tma_load_2d(b + bm * 128, &xmap, kb * kBK + kAtomK, m0, &full_bar[s]);
        ++issued;
      }
      if (!ok) {
        atomicOr(&flags, 2);
        // let every issued copy land before the CTA may exit
        for (int kb = (issued > stages ? issued - stages : 0); kb < issued; ++kb)
          mbar_wait_bounded(&full_bar[kb % stages], (kb / stages) & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issue (one lane)
    if (lane == 0) {
      const uint32_t idesc = idesc_f16(bm);
      bool ok = true;
      for (int kb = 0; kb < KT; ++kb) {
        const int s = kb % stages, use = kb / stages;
        if (!(ok = mbar_wait_bounded(&full_bar[s], use & 1))) break;
        tc_fence_after();
        const uint8_t *a = smem + s * L.stage_bytes + L.a_off;
        const uint8_t *b = smem + s * L.stage_bytes + L.b_off;
#pragma unroll
        for (int ks = 0; ks < kBK / 16; ++ks) {
          const int atom = ks / 4, kin = (ks % 4) * 32;  // bytes within the 128-byte row
          const uint64_t ad = sw128_desc(a + atom * (kBN * 128) + kin);
          const uint64_t bd = sw128_desc(b + atom * (bm * 128) + kin);
          mma_f16(tmem, ad, bd, idesc, (kb > 0 || ks > 0) ? 1u : 0u);
        }
        mma_commit(&empty_bar[s]);  // frees the stage once these MMAs have read it
      }
      if (!ok) atomicOr(&flags, 2);
      mma_commit(&accum_bar);  // the accumulator is final once every MMA above completes
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ dequant producers
    const int t = threadIdx.x - 128;            // column-row of the tile, 0..127
    const int b = (n0 >> 6) + (t >> 6);         // n-block of this row
    const int r = t & 63;                        // row inside the n-block
    const bool have = b < NB;                    // the last tile may have one n-block only
    const uint8_t *body = packed + kHeaderBytes + (size_t)(have ? b : 0) * KT * CB;
    const int gpc = kTileK / g;
    const int p = meta_pos(r);
    bool ok = true;
    // codes and meta of the next k-block are fetched one k-block ahead
    uint4 cw[4];
    uint32_t sc[4], zw[4];
    auto fetch = [&](int kb) {
      const uint8_t *ch = body + (size_t)kb * CB;
#pragma unroll
      for (int q = 0; q < 4; ++q) cw[q] = have ? __ldg(reinterpret_cast<const uint4 *>(ch + r * kRowBytes) + q)
                                            : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int l = 0; l < 4; ++l) {
        if (l < gpc && have) {
          const uint8_t *meta = ch + kCodeBytes + l * kGroupMetaBytes;
          sc[l] = __ldg(reinterpret_cast<const uint16_t *>(meta) + p);
          zw[l] = __ldg(reinterpret_cast<const uint32_t *>(meta + kScaleBytes) + p / 8);
        } else {
          sc[l] = 0;
          zw[l] = 0;
        }
      }
    };
    fetch(0);
    for (int kb = 0; kb < KT; ++kb) {
      const int s = kb % stages, use = kb / stages;
      uint4 c[4] = {cw[0], cw[1], cw[2], cw[3]};
      uint32_t scl[4] = {sc[0], sc[1], sc[2], sc[3]}, zl[4] = {zw[0], zw[1], zw[2], zw[3]};
      if (kb + 1 < KT) fetch(kb + 1);
      if (use > 0 && !(ok = mbar_wait_bounded(&empty_bar[s], (use - 1) & 1))) break;
      uint8_t *a = smem + s * L.stage_bytes + L.a_off;
      const uint32_t words[16] = {c[0].x, c[0].y, c[0].z, c[0].w, c[1].x, c[1].y, c[1].z, c[1].w,
                                  c[2].x, c[2].y, c[2].z, c[2].w, c[3].x, c[3].y, c[3].z, c[3].w};
#pragma unroll
      for (int w = 0; w < 16; ++w) {
        const int l = (8 * w) / g;  // group of these 8 k inside the chunk
        const ZeroBias zb = zero_bias((zl[l] >> (4 * (p % 8))) & 0xFu);
        const uint32_t s2 = scl[l] * 0x00010001u;
        uint32_t v[4];
        word_to_qz(words[w], zb, v);
        uint4 o;
        o.x = hmul2_u32(v[0], s2);
        o.y = hmul2_u32(v[1], s2);
        o.z = hmul2_u32(v[2], s2);
        o.w = hmul2_u32(v[3], s2);
        const int atom = w / 8, cc = w % 8;
        *reinterpret_cast<uint4 *>(a + atom * (kBN * 128) + t * 128 + ((cc ^ (t & 7)) << 4)) = o;
      }
      fence_proxy_async_smem();  // the tensor cores read this tile through the async proxy
      mbar_arrive(&full_bar[s]);
    }
    if (!ok) atomicOr(&flags, 2);
  }

  // ------------------------------------------------------------ epilogue: TMEM -> y (all warps)
  bool ok = mbar_wait_bounded(&accum_bar, 0);
  tc_fence_after();
  if (!ok) atomicOr(&flags, 2);
  griddep_wait();  // every storing thread waits for the previous kernel (a no-op once satisfied)
  if (threadIdx.x == 0) {
    const Header *h = reinterpret_cast<const Header *>(packed);
    if (h->magic != kMagic || h->version != kLayoutVersion || h->K != K || h->N != N || h->g != g) atomicOr(&flags, 1);
  }
  __syncthreads();
  const int fl = flags;
  if (!fl) {
    const int quarter = warp & 3, half = warp >> 2;
    const int n = n0 + 32 * quarter + lane;
    for (int c0 = 16 * half; c0 < bm; c0 += 32) {
      uint32_t v[16];
      tmem_ld16(tmem + ((uint32_t)(32 * quarter) << 16) + (uint32_t)c0, v);
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int m = m0 + c0 + j;
        if (m < M && n < N) y[(size_t)m * N + n] = __half_as_ushort(__float2half_rn(__uint_as_float(v[j])));
      }
    }
  } else if (threadIdx.x == 0) {
    atomicOr(err, fl);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(tmem_cols) : "memory");
  }
}

// --------------------------------------------------------------------------- host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void *p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

}  // namespace

int gemm_tc_block_m(int M) { return M >= 256 ? 256 : ((M + 15) / 16) * 16; }

cudaError_t launch_gemm_tc(const uint16_t *x, const void *packed, int M, int N, int K, int g, uint16_t *y, int *err,
                           cudaStream_t stream) {
  const int bm = gemm_tc_block_m(M);
  int stages = 0;
  while (stages < kMaxStages && gemm_smem(bm, stages + 1).total <= 200 * 1024) ++stages;
  const GemmSmem L = gemm_smem(bm, stages);
  int tmem_cols = 32;
  while (tmem_cols < bm) tmem_cols *= 2;

  auto enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  CUtensorMap map;
  const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
  const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kAtomK, (cuuint32_t)bm};
  const cuuint32_t es[2] = {1, 1};
  if (enc(&map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<uint16_t *>(x), dims, strides, box, es,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;

  static bool configured[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 210 * 1024);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((N + kBN - 1) / kBN, (M + bm - 1) / bm);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = L.total + 1024;  // + alignment slack
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemm_tc_kernel, map, static_cast<const uint8_t *>(packed), M, N, K, g,
                            num_ktiles(K), bm, stages, tmem_cols, y, err);
}

}  // namespace w4a16
