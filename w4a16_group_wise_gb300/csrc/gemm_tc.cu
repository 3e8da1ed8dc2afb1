// gemm_tc.cu -- tensor-core path of y = x . W for many rows of x (prefill).
//
// Why a second path: the CPU plugin found that a kernel which dequantizes once per row of
// activations is linear in the batch (12.9x slower than bf16 at 512 rows), so wide batches
// unpack the weight once and run an ordinary dense GEMM (vllm-omni commit "Add cpu_int4, an
// asymmetric 4-bit weight path for vLLM's CPU backend").  Here the unpacking is fused into the
// GEMM: each 128 x 128 weight tile is dequantized once per CTA into tensor memory and consumed
// by the 5th-generation tensor cores (tcgen05.mma, fp16 x fp16 -> fp32 in tensor memory); no
// dequantized W ever reaches HBM.
//
// Orientation: D[n][m] = sum_k W^T[n][k] * x^T[k][m], i.e. the MMA's M dimension (128) runs
// over output columns n and its N dimension (BM <= 256) over rows m of x, so few rows of x
// waste no tensor work.  Roles, per 128-k stage (one packed chunk) of a ring of up to 4 stages:
//  - one lane of warp 2 copies the packed chunks of the tile's two n-blocks (codes and their
//    scales and zeros, contiguous in the packed layout) into a ring of shared-memory slots with
//    bulk asynchronous copies, one 128-k chunk per slot;
//  - one lane of warp 0 loads the x tile (BM rows x 128 k, fp16) with two TMA copies into two
//    128-byte-swizzled K-major atoms of 64 k (rows past M and k past K read as 0);
//  - warps 4..11, in two groups taking the two 64-k halves of every stage (one lane per
//    column-row), read the codes from the slot, convert them to the exact fp16 weights
//    fp16((q - z) * s) (dq.cuh) and store them into the stage's A tile in tensor memory
//    (tcgen05.st);
//  - one lane of warp 1 issues 8 MMAs (K = 16 each, A from tensor memory, x from shared
//    memory) once both operands are in place and commits them to the stage's "empty" barrier,
//    which frees the stage when they complete.
// Without a K split the CTAs are persistent (one per SM, walking the tiles) and warps 12..15
// read each finished accumulator back (tcgen05.ld), round to fp16 and store y while the
// producers run ahead on the next tile; a CTA's last tile is drained by all 16 warps.  With a K
// split every CTA has one tile and all warps take part in adding the partial tiles.  The two
// cases run as separate instances of the kernel (PERSIST).  Every wait is bounded: on a timeout the kernel
// records an error, drains, frees tensor memory and skips the store.
// A bf16 layer runs the same kernel with T = Bf16 (dq.cuh): bf16 weights bf16((q - z) * s), x
// loaded as bf16 by the TMA, the bf16 operand type in the instruction descriptor, y rounded to
// bf16.
//
// Measured on GB300 while tuning this pipeline: keeping the A tile out of shared memory lets
// the ring hold 384 k at BM = 256; one warp's chain for 64 k (wait, read, convert, store,
// arrive) takes ~1200 cycles against ~670 cycles of MMAs, hence two converting groups; the
// MMA-issuing lane is on the critical path of every stage (~600 cycles of barrier wait, issue
// and commit per 4 MMAs), so its loop does no divisions and builds no descriptors, and a stage
// spans a whole chunk, so that one barrier round trip feeds 8 MMAs; and prefetching code chunks
// into L2 with bulk prefetches slowed the kernel once the rest was tuned (the copies compete
// for the same copy engine).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "../../include/w4a16.h"

#include "dq.cuh"
#include "bounds.cuh"
#include "kernels.h"
#include "layout.cuh"
#include "ptx.cuh"

namespace w4a16 {
namespace {

constexpr int kBN = 128;                      // weight rows (output columns n) per CTA = MMA M
constexpr int kBK = 64;                       // k per 128-byte swizzle atom of fp16
constexpr int kStageK = 128;                  // k per stage: one packed chunk, two atoms
constexpr int kMaxStages = 4;
// Tensor memory (512 columns x 128 lanes of 32 bits): the fp32 accumulator in columns
// [0, BM) -- or two, [0, BM) and [BM, 2 BM), so that a persistent CTA's epilogue drains one
// while the MMAs fill the other -- and the stages' fp16 A tiles (128 column-rows x 128 k = 64
// columns each) in the last 64 x stages columns.
constexpr int kTmemCols = 512;
// warp 0 x TMA, warp 1 MMA, warp 2 code copies, warps 4..11 dequant, warps 12..15 epilogue of a
// persistent CTA
constexpr int kThreads = 512;
constexpr int kDeqThreads = 256;
constexpr int kDeqWarps = kDeqThreads / 32;
constexpr int kEpiWarps = 4;
constexpr int kGroups = kThreads / 128;  // warps per TMEM lane quarter
constexpr int kMinCodeSlots = 3;      // 128-k chunks of codes in flight: at least this many,
constexpr int kMaxCodeSlots = 12;     // and as many as the shared memory left by the x stages holds
constexpr int kSmemBudget = 220 * 1024;
constexpr int kCodeSlotBytes = 9472;  // two n-blocks' chunks, 2 * (4096 + 4 * 160) at g = 32

struct GemmSmem {
  int stages, bm, cslots;
  int b_off, atom_bytes, stage_bytes, codes_off, epi_off, total;
};

// [stages x x-tile] [cslots x code slot], at least 32 KB (a one-tile CTA's epilogue reuses the
// front of it once the rings are idle), then 1 KB per persistent epilogue warp.  A stage's x tile is two swizzle atoms of
// BM rows x 64 k, the second at atom_bytes.  Small x tiles leave room for a deeper code ring:
// measured, the converting warps otherwise wait for the copies at small BM.
__host__ __device__ inline GemmSmem gemm_smem(int bm, int stages) {
  GemmSmem s;
  s.bm = bm;
  s.stages = stages;
  s.atom_bytes = bm * kBK * 2;
  s.stage_bytes = 2 * s.atom_bytes;
  s.b_off = 0;
  s.codes_off = stages * s.stage_bytes;
  int free_slots = (kSmemBudget - s.codes_off) / kCodeSlotBytes;
  s.cslots = free_slots < kMinCodeSlots ? kMinCodeSlots : free_slots > kMaxCodeSlots ? kMaxCodeSlots : free_slots;
  s.total = s.codes_off + s.cslots * kCodeSlotBytes;
  if (s.total < 32 * 1024) s.total = 32 * 1024;
  s.epi_off = s.total;  // the persistent epilogue's transpose buffers, 1 KB per warp
  s.total += kEpiWarps * 1024;
  return s;
}

// --------------------------------------------------------------------------- tcgen05 wrappers

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t sw128_desc(const void *p) {
  const uint64_t addr = smem_u32(p);
  return ((addr >> 4) & 0x3FFFull) | (1ull << 16) | (64ull << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor, kind::f16: fp16 A and B (K-major), fp32 D, M = 128, N = n; for a
// bf16 layer the A and B type fields (bits 7..9 and 10..12) hold 1, bf16.
template <class T>
__host__ __device__ inline uint32_t idesc_f16(int n) {
  const uint32_t ab = T::kDtype == kDtypeBf16 ? (1u << 7) | (1u << 10) : 0u;
  return (1u << 4) | ab | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}

// As mma_f16 with the A operand (128 rows x 16 k fp16, K-major) in tensor memory.
__device__ __forceinline__ void mma_f16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                               uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns from registers (one lane per thread of the warp),
// then wait until the stores are done.
__device__ __forceinline__ void tmem_st32_wait(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
      "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]),
      "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]),
      "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 lanes x 16 consecutive 32-bit columns (one lane per thread of the warp).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// global -> shared bulk copy (both 16-byte aligned, bytes a multiple of 16), completion as
// transaction bytes on `bar`.
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ uint32_t ld_cluster_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ float4 ld_cluster_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// As tmem_ld16 without the wait: several loads then one tmem_wait_ld.
__device__ __forceinline__ void tmem_ld16_async(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int c0, int c1, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(map), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}

// --------------------------------------------------------------------------- the kernel

// Split-K plan: each (n-tile, m-tile) is cut into `splits` consecutive ranges of 128-k stages.
// With splits > 1 the partial tiles are added in split order, so y does not depend on timing:
//  - cluster: the splits of a tile form one thread-block cluster; every CTA leaves its fp32
//    partial tile in its own shared memory and each adds a 1/splits slice of the tile from all
//    of them through distributed shared memory;
//  - global: every CTA stores its fp32 partial tile into the workspace and the last one to
//    finish a tile (per-tile arrival counter) adds the partials and writes y.
struct SplitPlan {
  int splits;
  int cluster;           // 1: cluster reduction, 0: workspace reduction
  int dbl;               // 1: two accumulators, alternating by tile (persistent CTAs)
  int a_col0;            // first tensor-memory column of the stages' A tiles
  int ntn, ntm;          // n-tiles and m-tiles of the problem
  int stages_per_split;  // 128-k stages per split (the last split may have fewer)
  float *partials;       // [splits][tiles][bm][128] fp32
  int *counters;         // [tiles], zero between calls
  long long partial_bytes;  // extent of `partials` (the bounds-checked build checks against it)
};

// Cluster split-K reduction of one CTA's pieces [e0, e1) of the tile (float4 pieces, 32 per row
// m): the S CTAs' fp32 partials (`part` in every CTA's shared memory), the other CTAs' read
// through distributed shared memory and this CTA's own (rank `me`) straight from its shared
// memory, added in rank order -- the workspace reduction's order -- and stored as y; U pieces per
// thread in flight.
template <class T, int S, int U>
__device__ __forceinline__ void cluster_reduce(const float *part, int me, int e0, int e1, int m0, int n0, int M,
                                               int N, uint16_t *__restrict__ y, int *err) {
  uint32_t base[S];
#pragma unroll
  for (int z = 0; z < S; ++z) base[z] = mapa_shared(part, (uint32_t)z);
  for (int e = e0 + (int)threadIdx.x; e < e1; e += U * kThreads) {
    float4 v[U][S];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int eu = e + u * kThreads;
      if (eu < e1) {
        const uint32_t off = (uint32_t)((eu >> 5) * kBN + 4 * (eu & 31)) * 4u;
#pragma unroll
        for (int z = 0; z < S; ++z)
          v[u][z] = z == me ? *reinterpret_cast<const float4 *>(reinterpret_cast<const uint8_t *>(part) + off)
                            : ld_cluster_f4(base[z] + off);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int eu = e + u * kThreads;
      if (eu >= e1) break;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int z = 0; z < S; ++z) {
        acc.x += v[u][z].x;
        acc.y += v[u][z].y;
        acc.z += v[u][z].z;
        acc.w += v[u][z].w;
      }
      const int gm = m0 + (eu >> 5), gn = n0 + 4 * (eu & 31);
      if (gm < M && gn < N && in_extent(y + (size_t)gm * N + gn, 8, y, 2LL * M * N, err)) {
        uint2 o;
        o.x = T::pack2(acc.x, acc.y);
        o.y = T::pack2(acc.z, acc.w);
        *reinterpret_cast<uint2 *>(y + (size_t)gm * N + gn) = o;
      }
    }
  }
}

template <class T, bool PERSIST>
__global__ void __launch_bounds__(kThreads, 1) gemm_tc_kernel(const __grid_constant__ CUtensorMap xmap,
                                                               const uint8_t *__restrict__ packed, int M, int N,
                                                               int K, int g, int KT, int bm, int stages,
                                                               int tmem_cols, SplitPlan sp, uint16_t *__restrict__ y,
                                                               int *err) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte alignment of the operand tiles (the swizzle pattern repeats every 1024 bytes)
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t full_bar[kMaxStages], empty_bar[kMaxStages], accum_bar;
  __shared__ uint64_t cfull_bar[kMaxCodeSlots], cempty_bar[kMaxCodeSlots];
  __shared__ uint64_t tfull_bar[2], tempty_bar[2];  // accumulator hand-offs of a persistent CTA
  __shared__ uint32_t tmem_base;
  __shared__ int flags, last;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const GemmSmem L = gemm_smem(bm, stages);
  const int NB = num_nblocks(N);
  const int CB = chunk_bytes(g);
  // buffer extents in bytes, for the bounds-checked build (x is read by TMA only, through a tensor
  // map of extent M x K: the copy engine fills coordinates outside it and reads nothing there)
  const long long pext = packed_extent(K, N, g), yext = 2LL * M * N;
  const int KS = KT;  // 128-k stages over K: one per chunk (k past K reads as 0 and has code 0)
  const int st_begin = blockIdx.z * sp.stages_per_split;
  const int nst = max(0, min(KS, st_begin + sp.stages_per_split) - st_begin);
  const uint32_t x_bytes = (uint32_t)L.stage_bytes;
  uint8_t *codes = smem + L.codes_off;
  // Tiles of this CTA: a persistent CTA takes tiles blockIdx.x, + gridDim.x, ... of the
  // (n-tile, m-tile) grid (m fastest, so neighbouring CTAs share weights); otherwise the one
  // tile (blockIdx.x, blockIdx.y).
  const int ntiles = sp.ntn * sp.ntm;
  const int my_tiles = PERSIST ? (ntiles - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x : 1;
  auto tile_n0 = [&](int it) {
    return (PERSIST ? ((int)blockIdx.x + it * (int)gridDim.x) / sp.ntm : (int)blockIdx.x) * kBN;
  };
  auto tile_m0 = [&](int it) {
    return (PERSIST ? ((int)blockIdx.x + it * (int)gridDim.x) % sp.ntm : (int)blockIdx.y) * bm;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full_bar[s], 1 + kDeqWarps);  // TMA expect-tx arrival + one per dequant warp
      mbar_init(&empty_bar[s], 1);             // one tcgen05.commit per use
    }
    for (int c = 0; c < L.cslots; ++c) {
      mbar_init(&cfull_bar[c], 1);             // expect-tx arrival of the bulk copies
      mbar_init(&cempty_bar[c], kDeqWarps);    // every dequant warp is done reading the slot
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull_bar[b], 1);             // one tcgen05.commit per tile
      mbar_init(&tempty_bar[b], kEpiWarps);    // every epilogue warp has read the accumulator
    }
    mbar_init(&accum_bar, 1);
    // the packed buffer must match the call (read-only: no need to wait for the previous kernel)
    const Header *h = reinterpret_cast<const Header *>(packed);
    flags = (!in_extent(h, sizeof(Header), packed, pext, err) || h->magic != kMagic ||
             h->version != kLayoutVersion || h->K != K || h->N != N || h->g != g || h->dtype != T::kDtype) ? 1 : 0;
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
  const bool run = flags == 0;  // a header mismatch writes nothing (same in every CTA)

  if (!run) {
    // nothing to do
  } else if (warp == 0) {
    // ------------------------------------------------------------ x tiles by TMA (one lane)
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(&xmap) : "memory");
      griddep_wait();  // x may be the previous kernel's output
      bool ok = true;
      int issued = 0;
      int s = 0, use = 0;
      for (int it = 0; it < my_tiles && ok; ++it) {
        const int m0 = tile_m0(it);
        for (int j = 0; j < nst; ++j) {
          if (use > 0 && !(ok = mbar_wait_sleep_bounded(&empty_bar[s], (use - 1) & 1))) break;
          mbar_arrive_expect_tx(&full_bar[s], x_bytes);
          uint8_t *xs = smem + s * L.stage_bytes + L.b_off;
          tma_load_2d(xs, &xmap, (st_begin + j) * kStageK, m0, &full_bar[s]);
          tma_load_2d(xs + L.atom_bytes, &xmap, (st_begin + j) * kStageK + kBK, m0, &full_bar[s]);
          ++issued;
          if (++s == stages) {
            s = 0;
            ++use;
          }
        }
      }
      if (!ok) {
        atomicOr(&flags, 2);
        // let every issued copy land before the CTA may exit
        for (int J = (issued > stages ? issued - stages : 0); J < issued; ++J)
          mbar_wait_bounded(&full_bar[J % stages], (J / stages) & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issue (one lane)
    if (lane == 0) {
      // This lane is on the critical path of every stage (measured: the MMAs of a stage take
      // ~670 cycles, and a loop with per-stage divisions and descriptor builds took ~1100), so
      // the ring position advances incrementally and the x descriptor is built once: its
      // start-address field counts 16-byte units, so a stage adds stage_bytes / 16 and a 16-k
      // step 2 and the second atom atom_bytes / 16 (shared addresses stay below 256 KB, so the
      // 14-bit field never carries).
      const uint32_t idesc = idesc_f16<T>(bm);
      const uint64_t bdesc0 = sw128_desc(smem + L.b_off);
      const uint32_t bstep = (uint32_t)L.stage_bytes >> 4;
      const uint64_t batom = (uint64_t)((uint32_t)L.atom_bytes >> 4);
      bool ok = true;
      int s = 0, use = 0;
      for (int it = 0; it < my_tiles && ok; ++it) {
        // accumulator ab is free once the epilogue warps have read the last tile that used it
        const int ab = sp.dbl ? (it & 1) : 0, ause = sp.dbl ? (it >> 1) : it;
        if (PERSIST && ause > 0 && !(ok = mbar_wait_sleep_bounded(&tempty_bar[ab], (ause - 1) & 1))) break;
        tc_fence_after();
        const uint32_t acc = tmem + (uint32_t)(ab * bm);
        for (int j = 0; j < nst; ++j) {
          if (!(ok = mbar_wait_sleep_bounded(&full_bar[s], use & 1))) break;
          tc_fence_after();
          const uint32_t a = tmem + (uint32_t)(sp.a_col0 + 64 * s);
          const uint64_t bd = bdesc0 + (uint64_t)(bstep * (uint32_t)s);
          mma_f16_tmem_a(acc, a, bd, idesc, j > 0 ? 1u : 0u);  // 16 k = 8 columns of A, 32 bytes of x
          mma_f16_tmem_a(acc, a + 8, bd + 2, idesc, 1u);
          mma_f16_tmem_a(acc, a + 16, bd + 4, idesc, 1u);
          mma_f16_tmem_a(acc, a + 24, bd + 6, idesc, 1u);
          mma_f16_tmem_a(acc, a + 32, bd + batom, idesc, 1u);  // second 64 k: the other atom
          mma_f16_tmem_a(acc, a + 40, bd + batom + 2, idesc, 1u);
          mma_f16_tmem_a(acc, a + 48, bd + batom + 4, idesc, 1u);
          mma_f16_tmem_a(acc, a + 56, bd + batom + 6, idesc, 1u);
          mma_commit(&empty_bar[s]);  // frees the stage once these MMAs have read it
          if (++s == stages) {
            s = 0;
            ++use;
          }
        }
        if (!ok) break;
        // the accumulator is final once every MMA above completes; the CTA's last tile goes to
        // all warps at the end, the others to the epilogue warps
        mma_commit(PERSIST && it + 1 < my_tiles ? &tfull_bar[ab] : &accum_bar);
      }
      if (!ok) {  // let every issued MMA finish before the CTA may exit
        atomicOr(&flags, 2);
        mma_commit(&accum_bar);
        mbar_wait_sleep_bounded(&accum_bar, 0);
      } else if (!mbar_wait_sleep_bounded(&accum_bar, 0)) {
        atomicOr(&flags, 2);
      }
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ packed chunks by bulk copy
    // (the packed weights are read-only: no need to wait for the previous kernel)
    if (lane == 0) {
      auto chunk_src = [&](int it, int lc, int q) {
        const int nb0 = tile_n0(it) >> 6;
        const uint8_t *src = packed + kHeaderBytes + ((size_t)(nb0 + q) * KT + st_begin + lc) * CB;
        return in_extent(src, CB, packed, pext, err) ? src : packed;  // a miss still completes the barrier
      };
      auto nblocks = [&](int it) { return ((tile_n0(it) >> 6) + 1 < NB) ? 2 : 1; };
      bool ok = true;
      int issued = 0;
      int cs = 0, use = 0;
      for (int it = 0; it < my_tiles && ok; ++it) {
        const int nblk = nblocks(it);
        for (int lc = 0; lc < nst; ++lc) {
          if (use > 0 && !(ok = mbar_wait_sleep_bounded(&cempty_bar[cs], (use - 1) & 1))) break;
          mbar_arrive_expect_tx(&cfull_bar[cs], (uint32_t)(nblk * CB));
          for (int q = 0; q < nblk; ++q)
            bulk_load(codes + cs * kCodeSlotBytes + q * CB, chunk_src(it, lc, q), (uint32_t)CB, &cfull_bar[cs]);
          ++issued;
          if (++cs == L.cslots) {
            cs = 0;
            ++use;
          }
        }
      }
      if (!ok) atomicOr(&flags, 2);
      // every issued copy has landed before the CTA may exit (at once in the normal case)
      for (int LC = (issued > L.cslots ? issued - L.cslots : 0); LC < issued; ++LC)
        mbar_wait_bounded(&cfull_bar[LC % L.cslots], (LC / L.cslots) & 1);
    }
  } else if (warp >= 4 && warp < 4 + kDeqWarps) {
    // ------------------------------------------------------------ dequant producers
    // Two groups of four warps take the two 64-k halves of every stage (group gsel: k 64 gsel ..
    // 64 gsel + 63 of each chunk), so both halves are converted at once and every chunk slot is
    // read by both groups.  In a group, lane l of warp w converts column-row r = 32 (w % 4) + l:
    // its 64 k are 32 code bytes of the row in the chunk slot (read one stage ahead, before the
    // waits, to hide the shared-memory latency), giving 32 columns of the stage's A tile.
    const int gsel = (warp - 4) >> 2;
    const int r = 32 * (warp & 3) + lane;
    const int gshift = g == 32 ? 5 : g == 64 ? 6 : 7;  // group of a 32-k span: (32 k32) >> gshift
    const int rr = r & 63;                        // row inside the n-block
    const int p = meta_pos(rr);
    const int rot = (rr >> 1) & 1;                // read order of the two 16-byte halves (banks)
    struct Codes {
      uint4 h[2];                                 // k 0..31 and 32..63 of the stage
      uint32_t sc[2], zw[2];                      // scale and zero word of each 32-k half
    };
    // read this group's half of a stage from code slot cs (have: the row's n-block exists)
    auto read_codes = [&](int cs, bool have, Codes &cd) {
      const uint8_t *ch = codes + cs * kCodeSlotBytes + (r >> 6) * CB;  // this row's chunk copy
      const int k64 = gsel;                                            // half of the chunk
      uint4 c0 = make_uint4(0, 0, 0, 0), c1 = c0;                      // read 0: half rot, read 1: the other
      uint32_t s0 = 0, s1 = 0, z0 = 0, z1 = 0;
      if (have) {
        const int ka = 2 * k64 + rot, kb = 2 * k64 + (rot ^ 1);
        const uint8_t *ma = ch + kCodeBytes + ((32 * ka) >> gshift) * kGroupMetaBytes;
        const uint8_t *mb = ch + kCodeBytes + ((32 * kb) >> gshift) * kGroupMetaBytes;
        c0 = *reinterpret_cast<const uint4 *>(ch + rr * kRowBytes + 16 * ka);
        c1 = *reinterpret_cast<const uint4 *>(ch + rr * kRowBytes + 16 * kb);
        s0 = *reinterpret_cast<const uint16_t *>(ma + 2 * p);
        s1 = *reinterpret_cast<const uint16_t *>(mb + 2 * p);
        z0 = *reinterpret_cast<const uint32_t *>(ma + kScaleBytes + 4 * (p / 8));
        z1 = *reinterpret_cast<const uint32_t *>(mb + kScaleBytes + 4 * (p / 8));
      }
      cd.h[0] = rot ? c1 : c0;
      cd.h[1] = rot ? c0 : c1;
      cd.sc[0] = rot ? s1 : s0;
      cd.sc[1] = rot ? s0 : s1;
      cd.zw[0] = rot ? z1 : z0;
      cd.zw[1] = rot ? z0 : z1;
    };
    auto row_has_block = [&](int it) { return (tile_n0(it) >> 6) + (r >> 6) < NB; };
    bool ok = true;
    Codes cur;
    int it = 0, j = 0;
    // ring positions, advanced incrementally: code slot of the current chunk and its use, stage
    // slot of the current stage and its use (one stage per chunk)
    int cs = 0, cuse = 0;
    int s = 0, use = 0;
    bool have = row_has_block(0);
    if (nst <= 0) it = my_tiles;
    if (it < my_tiles) {
      ok = mbar_wait_bounded(&cfull_bar[cs], cuse & 1);
      if (ok) read_codes(cs, have, cur);
    }
    while (it < my_tiles && ok) {
      // convert this stage's codes into registers
      uint4 out[8];
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const ZeroBias zb = T::zb((cur.zw[hh] >> (4 * (p % 8))) & 0xFu);
        const uint32_t s2 = cur.sc[hh] * 0x00010001u;
        const uint32_t words[4] = {cur.h[hh].x, cur.h[hh].y, cur.h[hh].z, cur.h[hh].w};
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          uint32_t v[4];
          T::qz(words[w], zb, v);
          out[4 * hh + w] = make_uint4(T::mul2(v[0], s2), T::mul2(v[1], s2), T::mul2(v[2], s2), T::mul2(v[3], s2));
        }
      }
      // every lane has its codes in registers: this group is done with the chunk's slot
      __syncwarp();
      if (lane == 0) mbar_arrive(&cempty_bar[cs]);
      // the group's next stage (the next chunk, or the first of the next tile): read it while
      // waiting for the stage buffer
      int itn = it, jn = j + 1;
      if (jn >= nst) {
        ++itn;
        jn = 0;
        if (itn < my_tiles) have = row_has_block(itn);
      }
      if (++cs == L.cslots) {
        cs = 0;
        ++cuse;
      }
      if (itn < my_tiles) {
        if (!(ok = mbar_wait_bounded(&cfull_bar[cs], cuse & 1))) break;
        read_codes(cs, have, cur);
      }
      if (use > 0 && !(ok = mbar_wait_bounded(&empty_bar[s], (use - 1) & 1))) break;
      tc_fence_after();  // after the MMAs that read this stage's A tile
      {
        // row r of the stage's A tile: lane r % 32 of the warp's lane quarter, 32 columns of
        // consecutive k pairs
        uint32_t v[32];
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) {
          v[4 * cc + 0] = out[cc].x;
          v[4 * cc + 1] = out[cc].y;
          v[4 * cc + 2] = out[cc].z;
          v[4 * cc + 3] = out[cc].w;
        }
        tmem_st32_wait(tmem + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)(sp.a_col0 + 64 * s + 32 * gsel), v);
      }
      tc_fence_before();  // the tensor cores read this tile after the barrier
      __syncwarp();
      if (lane == 0) mbar_arrive(&full_bar[s]);
      it = itn;
      j = jn;
      if (++s == stages) {
        s = 0;
        ++use;
      }
    }
    if (!ok) atomicOr(&flags, 2);
  } else if (warp >= 4 + kDeqWarps && PERSIST) {
    // ------------------------------------------------------------ persistent epilogue
    // Warp q of the four reads TMEM lanes 32q .. 32q + 31 (column-rows n) of an accumulator
    // (while the MMAs fill the other one, with two), 16 columns (rows m) at a time, rounds each
    // pair of rows into one fp16 pair and turns each 32 n x 16 m block around in its 1 KB of
    // shared memory, so that a lane stores 16 bytes of consecutive n of two rows m (measured:
    // the 4-byte stores of lane pairs this replaces took ~9,000 cycles per 256-row tile while the
    // MMAs waited).  The accumulator is released as soon as its last columns are in registers,
    // before they are stored (gate_up M = 512: 28.5 -> 26.7 us; M = 2048: 83 -> 78 us).
    const int q = warp & 3;
    uint16_t *th = reinterpret_cast<uint16_t *>(smem + L.epi_off + q * 1024);
    griddep_wait();  // y may still be read by the previous kernel
    bool ok = true;
    for (int it = 0; it + 1 < my_tiles && ok; ++it) {  // all but the last tile
      const int ab = sp.dbl ? (it & 1) : 0, ause = sp.dbl ? (it >> 1) : it;
      if (!(ok = mbar_wait_sleep_bounded(&tfull_bar[ab], ause & 1))) break;
      tc_fence_after();
      const int n0 = tile_n0(it) + 32 * q, m0 = tile_m0(it);
      const bool store = flags == 0;
      for (int c00 = 0; c00 < bm; c00 += 64) {  // four 16-column groups per wait
        uint32_t v[4][16];
#pragma unroll
        for (int b = 0; b < 4; ++b)
          if (c00 + 16 * b < bm)
            tmem_ld16_async(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(ab * bm + c00 + 16 * b), v[b]);
        tmem_wait_ld();
        if (c00 + 64 >= bm) {
          // the whole accumulator is in registers: the MMAs may refill it while the last
          // columns are stored
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&tempty_bar[ab]);
        }
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          if (c00 + 16 * b >= bm) break;
          // rows (2i, 2i + 1) of column-row n = lane as one fp16 pair, word n of row pair i (the
          // odd pairs with the two 4-word halves of each 8 n swapped, so that the 16-byte reads
          // below hit distinct banks)
          uint32_t *tw = reinterpret_cast<uint32_t *>(th);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            tw[i * 32 + (lane ^ (4 * (i & 1)))] = T::pack2(__uint_as_float(v[b][2 * i]), __uint_as_float(v[b][2 * i + 1]));
          __syncwarp();
          {  // lane: row pair i = lane / 4, n = 8 (lane % 4) .. + 7; rows 2i and 2i + 1 as 16-byte stores
            const int i = lane >> 2, nn = 8 * (lane & 3), sw = 4 * (i & 1);
            const uint4 a = *reinterpret_cast<const uint4 *>(tw + i * 32 + nn + sw);
            const uint4 c = *reinterpret_cast<const uint4 *>(tw + i * 32 + nn + (sw ^ 4));
            uint4 lo, hi;
            lo.x = __byte_perm(a.x, a.y, 0x5410);
            lo.y = __byte_perm(a.z, a.w, 0x5410);
            lo.z = __byte_perm(c.x, c.y, 0x5410);
            lo.w = __byte_perm(c.z, c.w, 0x5410);
            hi.x = __byte_perm(a.x, a.y, 0x7632);
            hi.y = __byte_perm(a.z, a.w, 0x7632);
            hi.z = __byte_perm(c.x, c.y, 0x7632);
            hi.w = __byte_perm(c.z, c.w, 0x7632);
            const int m = m0 + c00 + 16 * b + 2 * i, n = n0 + nn;
            if (store && m < M && n < N && in_extent(y + (size_t)m * N + n, 16, y, yext, err))
              *reinterpret_cast<uint4 *>(y + (size_t)m * N + n) = lo;
            if (store && m + 1 < M && n < N && in_extent(y + (size_t)(m + 1) * N + n, 16, y, yext, err))
              *reinterpret_cast<uint4 *>(y + (size_t)(m + 1) * N + n) = hi;
          }
          __syncwarp();
        }
      }
    }
    if (!ok) atomicOr(&flags, 2);
  }

  // ------------------------------------------------------------ epilogue of the CTA's last
  // (or only) tile, all warps.  Only the MMA lane waits for its accumulator (above); every other
  // thread parks in the hardware barrier below instead of polling, so the producers keep the
  // issue slots.  All 16 warps drain it (measured: a persistent CTA's last tile left to the four
  // epilogue warps kept the CTA alive ~7,600 cycles after its last MMA at BM = 256).
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (!run) {
    if (threadIdx.x == 0 && flags) atomicOr(err, flags);
  } else {
  griddep_wait();  // every storing thread waits for the previous kernel (a no-op once satisfied)
  const int n0 = tile_n0(my_tiles - 1), m0 = tile_m0(my_tiles - 1);
  const uint32_t acol = sp.dbl ? (uint32_t)(((my_tiles - 1) & 1) * bm) : 0u;  // its accumulator
  // Warp w reads TMEM lanes 32 (w % 4) .. + 31 (column-rows n) and the 16-column groups c of the
  // tile with c % kGroups == w / 4; a per-warp 2 KB transpose buffer in the (now idle) stage
  // memory turns each group into 16-byte stores of consecutive n.
  const int quarter = warp & 3, third = warp >> 2;
  const int nq = n0 + 32 * quarter;  // first column-row of this warp
  uint8_t *tb = smem + warp * 2048;
  const int tiles = gridDim.x * gridDim.y, tile = blockIdx.y * gridDim.x + blockIdx.x;
  int fl = flags;
  if (sp.cluster) {
    // partial tile [bm][128] fp32 in this CTA's (now idle) stage memory; the cluster is the
    // tile's splits, rank = blockIdx.z
    float *part = reinterpret_cast<float *>(smem);
    if (!fl) {
      for (int c00 = 16 * third; c00 < bm; c00 += 3 * 16 * kGroups) {  // three 16-column groups per wait
        uint32_t v[3][16];
#pragma unroll
        for (int b = 0; b < 3; ++b)
          if (c00 + 16 * kGroups * b < bm) tmem_ld16_async(tmem + ((uint32_t)(32 * quarter) << 16) + (uint32_t)(c00 + 16 * kGroups * b), v[b]);
        tmem_wait_ld();
#pragma unroll
        for (int b = 0; b < 3; ++b)
          if (c00 + 16 * kGroups * b < bm) {
#pragma unroll
            for (int j2 = 0; j2 < 16; ++j2)
              part[(c00 + 16 * kGroups * b + j2) * kBN + 32 * quarter + lane] = __uint_as_float(v[b][j2]);
          }
      }
    }
    cluster_arrive();  // release: partials and flags of every CTA are visible to the cluster
    cluster_wait();
    int any = 0;
    for (int z = 0; z < sp.splits; ++z) any |= (int)ld_cluster_u32(mapa_shared(&flags, (uint32_t)z));
    if (any) {
      if (blockIdx.z == 0 && threadIdx.x == 0) atomicOr(err, any);
    } else {
      const int E = bm * (kBN / 4);  // float4 pieces of the tile, 32 per row m
      const int me = (int)blockIdx.z;  // rank in the cluster (1 x 1 x splits)
      const int e0 = (int)((long)blockIdx.z * E / sp.splits), e1 = (int)((long)(blockIdx.z + 1) * E / sp.splits);
      // pieces in flight per thread: 16 loads whatever the split count (measured: two pieces per
      // thread, four round trips at two splits, took ~5,600 cycles per 256-row tile)
      switch (sp.splits) {
        case 2: cluster_reduce<T, 2, 8>(part, me, e0, e1, m0, n0, M, N, y, err); break;
        case 3: cluster_reduce<T, 3, 5>(part, me, e0, e1, m0, n0, M, N, y, err); break;
        case 4: cluster_reduce<T, 4, 4>(part, me, e0, e1, m0, n0, M, N, y, err); break;
        case 5: cluster_reduce<T, 5, 3>(part, me, e0, e1, m0, n0, M, N, y, err); break;
        case 6: cluster_reduce<T, 6, 2>(part, me, e0, e1, m0, n0, M, N, y, err); break;
        case 7: cluster_reduce<T, 7, 2>(part, me, e0, e1, m0, n0, M, N, y, err); break;
        default: cluster_reduce<T, 8, 2>(part, me, e0, e1, m0, n0, M, N, y, err); break;
      }
    }
    cluster_arrive();  // no CTA leaves while another still reads its partial
    cluster_wait();
  } else if (sp.splits > 1) {
    // store this split's fp32 partial tile [bm][128], then count the arrival
    float *mine = sp.partials + ((size_t)blockIdx.z * tiles + tile) * bm * kBN;
    if (!fl) {
      for (int c0 = 16 * third; c0 < bm; c0 += 16 * kGroups) {
        uint32_t v[16];
        tmem_ld16(tmem + ((uint32_t)(32 * quarter) << 16) + (uint32_t)c0, v);
#pragma unroll
        for (int j2 = 0; j2 < 16; ++j2) reinterpret_cast<uint32_t *>(tb)[j2 * 32 + lane] = v[j2];
        __syncwarp();
#pragma unroll
        for (int q = 0; q < 4; ++q) {  // 128 pieces of 4 floats: (m = piece / 8, n = 4 * (piece % 8))
          const int pc = lane + 32 * q, j2 = pc >> 3, nn = 4 * (pc & 7);
          float *dst = mine + (size_t)(c0 + j2) * kBN + 32 * quarter + nn;
          if (in_extent(dst, 16, sp.partials, sp.partial_bytes, err))
            __stcg(reinterpret_cast<float4 *>(dst), *reinterpret_cast<const float4 *>(tb + (j2 * 32 + nn) * 4));
        }
        __syncwarp();
      }
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0)
      last = in_extent(&sp.counters[tile], 4, sp.counters, (long long)kSplitCounterBytes, err) &&
             (atomicAdd(&sp.counters[tile], 1) == sp.splits - 1);
    __syncthreads();
    if (!last) {
      if (fl && threadIdx.x == 0) atomicOr(err, fl);  // the last CTA adds what it finds
      fl = 0;
    } else {
      __threadfence();
      if (threadIdx.x == 0) sp.counters[tile] = 0;  // ready for the next call
    }
  }
  if (sp.cluster || (sp.splits > 1 && !last)) {
    // nothing more to do
  } else if (fl) {
    if (threadIdx.x == 0) atomicOr(err, fl);
  } else if (sp.splits > 1) {
    // add the partials in split order, 4 consecutive n per piece
    for (int c0 = 16 * third; c0 < bm; c0 += 16 * kGroups) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int pc = lane + 32 * q, j2 = pc >> 3, nn = 4 * (pc & 7);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int z = 0; z < sp.splits; ++z) {
          const float *src = sp.partials + (((size_t)z * tiles + tile) * bm + c0 + j2) * kBN + 32 * quarter + nn;
          const float4 v = in_extent(src, 16, sp.partials, sp.partial_bytes, err)
                               ? __ldcg(reinterpret_cast<const float4 *>(src)) : make_float4(0.f, 0.f, 0.f, 0.f);
          acc.x += v.x;
          acc.y += v.y;
          acc.z += v.z;
          acc.w += v.w;
        }
        const int m = m0 + c0 + j2, n = nq + nn;
        if (m < M && n < N && in_extent(y + (size_t)m * N + n, 8, y, yext, err)) {
          uint2 o;
          o.x = T::pack2(acc.x, acc.y);
          o.y = T::pack2(acc.z, acc.w);
          *reinterpret_cast<uint2 *>(y + (size_t)m * N + n) = o;
        }
      }
    }
  } else {
    // rows (2i, 2i + 1) of a 16-column group as fp16 pairs, turned around as in the persistent
    // epilogue: 16-byte stores of 8 consecutive n of two rows
    uint32_t *tw = reinterpret_cast<uint32_t *>(tb);
    for (int c00 = 16 * third; c00 < bm; c00 += 3 * 16 * kGroups) {  // three 16-column groups per wait
      uint32_t v[3][16];
#pragma unroll
      for (int b = 0; b < 3; ++b)
        if (c00 + 16 * kGroups * b < bm)
          tmem_ld16_async(tmem + ((uint32_t)(32 * quarter) << 16) + acol + (uint32_t)(c00 + 16 * kGroups * b), v[b]);
      tmem_wait_ld();
#pragma unroll
      for (int b = 0; b < 3; ++b) {
        const int c0 = c00 + 16 * kGroups * b;
        if (c0 >= bm) break;
#pragma unroll
        for (int i = 0; i < 8; ++i)
          tw[i * 32 + (lane ^ (4 * (i & 1)))] = T::pack2(__uint_as_float(v[b][2 * i]), __uint_as_float(v[b][2 * i + 1]));
        __syncwarp();
        {
          const int i = lane >> 2, nn = 8 * (lane & 3), sw = 4 * (i & 1);
          const uint4 a = *reinterpret_cast<const uint4 *>(tw + i * 32 + nn + sw);
          const uint4 c = *reinterpret_cast<const uint4 *>(tw + i * 32 + nn + (sw ^ 4));
          uint4 lo, hi;
          lo.x = __byte_perm(a.x, a.y, 0x5410);
          lo.y = __byte_perm(a.z, a.w, 0x5410);
          lo.z = __byte_perm(c.x, c.y, 0x5410);
          lo.w = __byte_perm(c.z, c.w, 0x5410);
          hi.x = __byte_perm(a.x, a.y, 0x7632);
          hi.y = __byte_perm(a.z, a.w, 0x7632);
          hi.z = __byte_perm(c.x, c.y, 0x7632);
          hi.w = __byte_perm(c.z, c.w, 0x7632);
          const int m = m0 + c0 + 2 * i, n = nq + nn;
          if (m < M && n < N && in_extent(y + (size_t)m * N + n, 16, y, yext, err))
            *reinterpret_cast<uint4 *>(y + (size_t)m * N + n) = lo;
          if (m + 1 < M && n < N && in_extent(y + (size_t)(m + 1) * N + n, 16, y, yext, err))
            *reinterpret_cast<uint4 *>(y + (size_t)(m + 1) * N + n) = hi;
        }
        __syncwarp();
      }
    }
  }
  }  // one-tile epilogue
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(tmem_cols) : "memory");
  }
}

// --------------------------------------------------------------------------- host side

}  // namespace

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
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

namespace {

int sm_count_tc() {
  static std::atomic<int> count[64];  // per device, 0 until looked up
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return 148;
  int n = count[dev].load(std::memory_order_relaxed);
  if (!n) {
    int c = 0;
    cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev);
    n = c > 0 ? c : 148;
    count[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

// Workspace of a split-K launch with the workspace reduction: kCounterBytes of per-tile
// arrival counters at offset 0 (zero before the first call, left zero by every completed call,
// whatever the shape), then the fp32 partial tiles (no initialisation needed).
constexpr int kCounterBytes = (int)kSplitCounterBytes;
constexpr int kMaxSplitTiles = kCounterBytes / 4;
constexpr int kMaxSplits = 8;            // portable cluster size
constexpr int kSmemLimit = 226 * 1024;   // opt-in dynamic shared memory of the kernel (+1 KB static)

// Stages that fit both the shared memory (x ring and code slots) and the tensor memory left by
// the accumulators.
int fit_stages(int bm, bool dbl) {
  const int acc = dbl ? 2 * bm : bm;
  int st = 0;
  while (st < kMaxStages && gemm_smem(bm, st + 1).epi_off <= kSmemBudget && acc + 64 * (st + 1) <= kTmemCols) ++st;
  return st;
}

std::atomic<int> g_splitk_mode{W4A16_SPLITK_AUTO};

// How many clusters of `splits` CTAs of this kernel can be resident at once on the current
// device (every configuration holds one CTA per SM); cached per device and cluster size.
int max_clusters(int splits) {
  static std::mutex mu;
  static int cache[64][kMaxSplits + 1];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || splits < 1 || splits > kMaxSplits) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev][splits]) {
    int n = 0;
    if (cudaFuncSetAttribute(gemm_tc_kernel<Fp16, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit) == cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(1, 1, splits);
      cfg.blockDim = dim3(kThreads);
      cfg.dynamicSmemBytes = kSmemLimit;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 1;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = splits;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      if (cudaOccupancyMaxActiveClusters(&n, gemm_tc_kernel<Fp16, false>, &cfg) != cudaSuccess) n = 0;
    }
    cudaGetLastError();
    cache[dev][splits] = n > 0 ? n : -1;
  }
  return cache[dev][splits] > 0 ? cache[dev][splits] : 0;
}

}  // namespace

TcPlan plan_gemm_tc(int M, int N, int K) {
  TcPlan p;
  const int ntn = (N + kBN - 1) / kBN;
  const int KS = num_ktiles(K);  // 128-k stages
  const int sms = sm_count_tc();
  p.bm = M >= 256 ? 256 : ((M + 15) / 16) * 16;
  p.dbl = false;
  p.tmem_cols = kTmemCols;
  int tiles = ntn * ((M + p.bm - 1) / p.bm);
  // Too few 256-row tiles to cover the GPU, but enough 128-row tiles to cover half of it in one
  // round: take the half-height tiles and no K split.  Measured at M = 512: q_k_v (48 tiles at
  // BM = 256, two K splits) went from 14.4 to 13.2 us with 96 whole-K tiles; down (32 tiles, four
  // splits) went from 19.5 to 21.5 us with 64 half-height tiles and two splits, so there BM stays
  // 256.  A second round of half-height tiles costs more than it saves: a 128-row stage takes
  // ~1300 cycles against ~1400 for 256 rows (q_k_v M = 1024: 20.9 us with 192 tiles of 128 rows,
  // 15.4 us with 96 of 256).
  if (p.bm == 256 && 4 * tiles < 3 * sms) {
    const int tiles128 = ntn * ((M + 127) / 128);
    if (2 * tiles128 >= sms && tiles128 <= sms) {
      p.bm = 128;
      tiles = tiles128;
    }
  }
  // Split K when the tiles alone would leave a quarter of the SMs or more idle; keep at least
  // two 128-k stages per split and at most one cluster's worth of splits.  Where the device runs
  // clusters, all clusters of the launch must be resident at once (measured: a second wave of
  // clusters costs more than the splits gain), so the split count is lowered until they are;
  // both reductions use the same count, so they add the same partial tiles.
  const int mode = g_splitk_mode.load();
  const bool clusters = max_clusters(2) > 0;
  p.splits = 1;
  if (4 * tiles < 3 * sms && tiles <= kMaxSplitTiles) {
    p.splits = sms / tiles;
    if (p.splits > KS / 2) p.splits = KS / 2;
    if (p.splits > kMaxSplits) p.splits = kMaxSplits;
    if (p.splits < 1) p.splits = 1;
    if (clusters)
      while (p.splits > 1 && max_clusters(p.splits) < tiles) --p.splits;
  }
  // Persistent CTAs (no split) alternate two accumulators when both fit in tensor memory beside
  // the A stages (BM <= 160), so that a tile's drain overlaps the next tile's MMAs.  Larger M
  // keeps BM = 256 and one accumulator: measured, one tcgen05.mma takes the issuing lane ~90
  // cycles, so the 64-cycle MMAs of BM = 128 left the tensor pipe idle (gate_up M = 2048: 109 us
  // against 84 us at BM = 256).
  if (p.splits == 1) p.dbl = p.bm <= 160;
  p.tiles = tiles;
  p.stages = fit_stages(p.bm, p.dbl);
  p.a_col0 = kTmemCols - 64 * p.stages;
  p.stages_per_split = (KS + p.splits - 1) / p.splits;
  p.splits = (KS + p.stages_per_split - 1) / p.stages_per_split;  // no empty split
  p.cluster = p.splits > 1 && mode != W4A16_SPLITK_GLOBAL && clusters && max_clusters(p.splits) >= p.tiles;
  p.partial_bytes = (p.splits > 1 && !p.cluster) ? (size_t)p.splits * p.tiles * p.bm * kBN * sizeof(float) : 0;
  p.persist = p.splits == 1;
  if (!p.persist) p.dbl = false;
  return p;
}

size_t gemm_tc_workspace_bytes(const TcPlan &p) { return p.partial_bytes ? kCounterBytes + p.partial_bytes : 0; }

int set_splitk_mode(int mode) {
  if (mode != W4A16_SPLITK_AUTO && mode != W4A16_SPLITK_GLOBAL) return W4A16_ERR_INVALID;
  g_splitk_mode.store(mode);
  return W4A16_OK;
}

namespace {

// The TMA map of x (K-major, 128-byte swizzle, boxes of 64 k x bm rows; zero fill past M and K).
// Encoding one costs a driver call, so each host thread keeps the last few it made, keyed by
// everything the map depends on; a call with the same x buffer and shape reuses it.
template <class T>
bool x_tensor_map(CUtensorMap &map, const uint16_t *x, int M, int K, int bm) {
  struct Entry {
    const void *x;
    int M, K, bm, dtype;
    CUtensorMap map;
  };
  constexpr int kEntries = 8;
  thread_local Entry cache[kEntries];
  thread_local int next = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  const int key_dtype = T::kDtype * 256 + dev;  // the element type and the device
  for (int i = 0; i < kEntries; ++i) {
    const Entry &e = cache[i];
    if (e.x == x && e.M == M && e.K == K && e.bm == bm && e.dtype == key_dtype) {
      map = e.map;
      return true;
    }
  }
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
  const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)bm};
  const cuuint32_t es[2] = {1, 1};
  const CUtensorMapDataType xtype = T::kDtype == kDtypeBf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  if (enc(&map, xtype, 2, const_cast<uint16_t *>(x), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  Entry &e = cache[next];
  next = (next + 1) % kEntries;
  e = Entry{x, M, K, bm, key_dtype, map};
  return true;
}

template <class T>
cudaError_t launch_gemm_tc_t(const TcPlan &P, const uint16_t *x, const void *packed, int M, int N, int K, int g,
                             uint16_t *y, int *err, void *workspace, cudaStream_t stream) {
  const GemmSmem L = gemm_smem(P.bm, P.stages);

  CUtensorMap map;
  if (!x_tensor_map<T>(map, x, M, K, P.bm)) return cudaErrorInvalidValue;

  SplitPlan sp;
  sp.splits = P.splits;
  sp.cluster = P.cluster ? 1 : 0;
  sp.stages_per_split = P.stages_per_split;
  sp.dbl = P.dbl ? 1 : 0;
  sp.a_col0 = P.a_col0;
  sp.ntn = (N + kBN - 1) / kBN;
  sp.ntm = (M + P.bm - 1) / P.bm;
  const bool global = P.partial_bytes > 0;
  sp.counters = global ? static_cast<int *>(workspace) : nullptr;
  sp.partials = global ? reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + kCounterBytes) : nullptr;
  sp.partial_bytes = (long long)P.partial_bytes;

  // Persistent and split-K launches run separate instances of the kernel, each compiled without
  // the other's epilogue (measured: with both in one function, adding work to the persistent
  // epilogue slowed the split-K shapes by 1-3%).
  auto kernel = P.persist ? gemm_tc_kernel<T, true> : gemm_tc_kernel<T, false>;
  static std::atomic<bool> configured[2][64];  // per instance and device: the attribute has been set
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !configured[P.persist][dev].load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
    if (e != cudaSuccess) return e;
    configured[P.persist][dev].store(true, std::memory_order_release);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = P.persist ? dim3(std::min(P.tiles, sm_count_tc())) : dim3(sp.ntn, sp.ntm, P.splits);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = L.total + 1024;  // + alignment slack
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  int na = 1;
  if (P.cluster) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 1;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = P.splits;
    na = 2;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, kernel, map, static_cast<const uint8_t *>(packed), M, N, K, g,
                            num_ktiles(K), P.bm, P.stages, P.tmem_cols, sp, y, err);
}

}  // namespace

cudaError_t launch_gemm_tc(const TcPlan &plan, const uint16_t *x, const void *packed, int M, int N, int K, int g,
                           int dtype, uint16_t *y, int *err, void *workspace, cudaStream_t stream) {
  if (plan.partial_bytes > 0 && !workspace) return cudaErrorInvalidValue;
  return dtype == kDtypeBf16 ? launch_gemm_tc_t<Bf16>(plan, x, packed, M, N, K, g, y, err, workspace, stream)
                             : launch_gemm_tc_t<Fp16>(plan, x, packed, M, N, K, g, y, err, workspace, stream);
}

}  // namespace w4a16
