// gemv.cu -- decode path of y = x . W for few rows of x (M <= 32).
//
// Four kernels, picked by launch_gemv from M, K and the number of 16-column row-tiles:
// gemv_kernel (M <= 16, x in registers), gemv_small_kernel (M <= 8, x through a per-warp cp.async
// ring, 64-80 registers so that 3-4 CTAs fit per SM), gemv_stream_kernel (M <= 8, K <= 2048 and
// very wide layers: resident CTAs walking row-tile pairs) and gemv_mid_kernel (17 <= M <= 32: x
// staged once per CTA, K split over a cluster).
// What follows holds for all four.
//
// Why a separate path: "single-stream decode reads every weight to emit one token, so bits
// per weight set the token rate" (vllm-omni commit "Add cpu_int4, an asymmetric 4-bit weight
// path for vLLM's CPU backend").  The kernel streams the packed weights exactly once, with
// enough bytes in flight for HBM and as little fixed latency per launch as possible:
//  - one CTA owns RT row-tiles (16 columns each) of one 64-column n-block over the whole of K,
//    so there is no reduction across CTAs; its W warps take the 128-k chunks round-robin;
//  - every lane loads its codes with 16-byte non-allocating loads (a warp's load covers 8
//    column-rows x 128 k = 512 contiguous bytes), software-pipelined about 4 KB deep per warp;
//    the weights are requested before waiting on the previous kernel in the stream
//    (programmatic dependent launch: they are read-only);
//  - x (L1-cached loads, zero past M and K) is fetched one chunk ahead of its use (staging it
//    in shared memory first was measured slower: every warp then waits for all of x);
//  - nibbles are converted to fp16 in registers (dq.cuh) and the tensor pipe does the
//    multiply-adds (mma.sync m16n8k16, fp16 x fp16 -> fp32), so the CUDA cores only issue the
//    conversion.  The weight tile is the A operand (16 columns n x 16 k) and x^T the B operand
//    (16 k x 8 rows m): M <= 8 costs one MMA per 256 weights, M <= 16 two.
// (Bulk asynchronous copies of the weights into shared memory were measured slower here: the
// copies of one CTA complete about one at a time, so a CTA's stream is latency-bound unless
// each copy is tens of KB.)
//
// k permutation inside a 128-k chunk: lane (r8 = lane/4, t = lane%4) owns the 32-k span
// [32t, 32t+32) of its column-rows; MMA step j maps the fragment's logical k {2t, 2t+1, 2t+8,
// 2t+9} to physical k 32t + 4j + {0, 1, 2, 3}.  A and B fragments both index k by t, so the
// products are unchanged and every lane reads contiguous data.
//
// Scale: for g = 128 a chunk is one group, so each chunk's MMA chains sum (q - z) * x exactly in
// fp32 and the fp32 scale is applied once per (column, row of x) at the end of the chunk.  For
// g = 32 / 64 a chain spans several groups and each weight is multiplied by its scale in fp16
// (the exact fp16 weight) before the MMA.
//
// The warps' partial sums are added in warp order through shared memory, so y is bit-identical
// from run to run.
//
// Every kernel is instantiated for fp16 and for bf16 layers (T = Fp16 / Bf16 of dq.cuh: the
// nibble conversion, the scale multiply, the mma.sync operand type and the output rounding).
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>

#include "bounds.cuh"
#include "dq.cuh"
#include "kernels.h"
#include "layout.cuh"
#include "ptx.cuh"

namespace w4a16 {
namespace {

constexpr int kMaxWarps = 16;

__device__ __forceinline__ uint4 ld_stream16(const void *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t ld_stream4(const void *p) {
  uint32_t v;
  asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t ld_stream1(const void *p) {
  uint16_t v;
  asm volatile("ld.global.nc.L1::no_allocate.u8 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

// The loads of the packed weights, through the debug build's bounds check (bounds.cuh): pext is
// the packed buffer's extent in bytes.
__device__ __forceinline__ uint4 ld_w16(const uint8_t *p, const uint8_t *packed, long long pext, int *err) {
  return in_extent(p, 16, packed, pext, err) ? ld_stream16(p) : make_uint4(0, 0, 0, 0);
}
__device__ __forceinline__ uint32_t ld_w4(const uint8_t *p, const uint8_t *packed, long long pext, int *err) {
  return in_extent(p, 4, packed, pext, err) ? ld_stream4(p) : 0u;
}
__device__ __forceinline__ uint32_t ld_w1(const uint8_t *p, const uint8_t *packed, long long pext, int *err) {
  return in_extent(p, 1, packed, pext, err) ? ld_stream1(p) : 0u;
}
// The header check of a kernel (thread 0): the buffer describes this layer.
template <class T>
__device__ __forceinline__ int header_ok(const uint8_t *packed, int K, int N, int g, long long pext, int *err) {
  if (!in_extent(packed, sizeof(Header), packed, pext, err)) return 0;
  const Header *h = reinterpret_cast<const Header *>(packed);
  return (h->magic == kMagic) & (h->version == kLayoutVersion) & (h->K == K) & (h->N == N) & (h->g == g) &
         (h->dtype == T::kDtype);
}

// What one lane holds for one chunk of weights.
template <int RT>
struct Stage {
  uint4 code[RT][2];   // [row-tile][rows r8, r8 + 8], 32 k each
  uint32_t scale[RT];  // scales of rows r8 (low half) and r8 + 8 (high half)
  uint32_t zero[RT];   // zero codes: bits 0..3 row r8, bits 4..7 row r8 + 8
};

// x[m][32 k of the lane's span], m = m0 + r8 (+ 8); zeros past M or K
template <int MB>
struct XFrag {
  uint4 v[MB][4];
};

// RT: row-tiles per CTA (1 or 2).  MB: 8-row blocks of x (1: M <= 8, 2: M <= 16).  FACTOR:
// scale applied per chunk in fp32 (g == 128) instead of per weight in fp16.
// Sixteen warps are only launched for RT == 1, MB == 1; the other variants get more registers.
template <int RT, int MB>
constexpr int kThreadBound = (RT == 1 && MB == 1) ? kMaxWarps * 32 : kMaxWarps * 16;

template <class T, int RT, int MB, bool FACTOR>
__global__ void __launch_bounds__(kThreadBound<RT, MB>) gemv_kernel(const uint16_t *__restrict__ x,
                                                              const uint8_t *__restrict__ packed, int M, int N,
                                                              int K, int g, int KT, uint16_t *__restrict__ y,
                                                              int *err) {
  constexpr int kDepth = 4 / RT;      // chunks of weights in flight per warp (~4 KB); even
  constexpr int kVals = RT * MB * 4;  // accumulator values per lane
  extern __shared__ __align__(16) float red[];  // [W][kVals][32]
  __shared__ int bad;

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, W = blockDim.x >> 5;
  const int r8 = lane >> 2, t = lane & 3;
  const int tile0 = blockIdx.x * RT;  // first row-tile (16 columns) of this CTA
  const int b = tile0 / 4, i0 = tile0 % 4;
  const int m0 = blockIdx.y * 8 * MB;
  const int CB = chunk_bytes(g);
  const uint8_t *body = packed + kHeaderBytes + (size_t)b * KT * CB;
  const int mine = (KT - warp + W - 1) / W;  // chunks warp, warp + W, ...

  const long long pext = packed_extent(K, N, g), xext = 2LL * M * K, yext = 2LL * M * N;
  int hdr_ok = 1;
  if (threadIdx.x == 0) hdr_ok = header_ok<T>(packed, K, N, g, pext, err);  // checked at the end

  auto load_w = [&](Stage<RT> &st, int j) {
    const uint8_t *ch = body + (size_t)(warp + j * W) * CB;
    const uint8_t *meta = ch + kCodeBytes + ((32 * t) / g) * kGroupMetaBytes;
#pragma unroll
    for (int r = 0; r < RT; ++r) {
      const int i = i0 + r;
#pragma unroll
      for (int h = 0; h < 2; ++h)
        st.code[r][h] = ld_w16(ch + (16 * i + r8 + 8 * h) * kRowBytes + 16 * t, packed, pext, err);
      st.scale[r] = ld_w4(meta + 2 * (8 * r8 + 2 * i), packed, pext, err);
      st.zero[r] = ld_w1(meta + kScaleBytes + 4 * r8 + i, packed, pext, err);
    }
  };
  auto load_x = [&](XFrag<MB> &xf, int j) {
    const int kx = (warp + j * W) * kTileK + 32 * t;
#pragma unroll
    for (int mb = 0; mb < MB; ++mb) {
      const int m = m0 + 8 * mb + r8;
      const bool in = (m < M) && (kx < K) && in_extent(x + (size_t)m * K + kx, 64, x, xext, err);
      const uint4 *xp = reinterpret_cast<const uint4 *>(x + (size_t)(in ? m : 0) * K + (in ? kx : 0));
#pragma unroll
      for (int q = 0; q < 4; ++q) xf.v[mb][q] = in ? __ldg(xp + q) : make_uint4(0, 0, 0, 0);
    }
  };

  float acc[RT][MB][4];
#pragma unroll
  for (int r = 0; r < RT; ++r)
#pragma unroll
    for (int mb = 0; mb < MB; ++mb)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[r][mb][c] = 0.f;

  Stage<RT> st[kDepth];
  XFrag<MB> xa, xb;  // x of the current and the next chunk, alternating
#pragma unroll
  for (int d = 0; d < kDepth; ++d)
    if (d < mine) load_w(st[d], d);
  griddep_launch_dependents();
  griddep_wait();  // x may be the previous kernel's output; y may still be read by it
  if (mine > 0) load_x(xa, 0);

#pragma unroll 1
  for (int j0 = 0; j0 < mine; j0 += kDepth) {
#pragma unroll
    for (int d = 0; d < kDepth; ++d) {
      const int j = j0 + d;
      if (j < mine) {
        XFrag<MB> &xc = (d & 1) ? xb : xa;
        XFrag<MB> &xn = (d & 1) ? xa : xb;
        if (j + 1 < mine) load_x(xn, j + 1);
        Stage<RT> &s = st[d];
#pragma unroll
        for (int r = 0; r < RT; ++r) {
          const ZeroBias zb0 = T::zb(s.zero[r] & 0xFu), zb1 = T::zb((s.zero[r] >> 4) & 0xFu);
          float dd[MB][4];
#pragma unroll
          for (int mb = 0; mb < MB; ++mb)
#pragma unroll
            for (int e = 0; e < 4; ++e) dd[mb][e] = 0.f;
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            const uint32_t w0 = (w == 0) ? s.code[r][0].x : (w == 1) ? s.code[r][0].y : (w == 2) ? s.code[r][0].z : s.code[r][0].w;
            const uint32_t w1 = (w == 0) ? s.code[r][1].x : (w == 1) ? s.code[r][1].y : (w == 2) ? s.code[r][1].z : s.code[r][1].w;
            uint32_t v0[4], v1[4];
            T::qz(w0, zb0, v0);
            T::qz(w1, zb1, v1);
            if (!FACTOR) {
              const uint32_t s20 = (s.scale[r] & 0xFFFFu) * 0x00010001u, s21 = (s.scale[r] >> 16) * 0x00010001u;
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                v0[e] = T::mul2(v0[e], s20);
                v1[e] = T::mul2(v1[e], s21);
              }
            }
#pragma unroll
            for (int mb = 0; mb < MB; ++mb) {
              float *dst = FACTOR ? dd[mb] : acc[r][mb];
              const uint4 xw = xc.v[mb][w];
              T::mma16816(dst, v0[0], v1[0], v0[1], v1[1], xw.x, xw.y);  // k 8w + 0..3
              T::mma16816(dst, v0[2], v1[2], v0[3], v1[3], xw.z, xw.w);  // k 8w + 4..7
            }
          }
          if (FACTOR) {
            const float f0 = T::to_float(s.scale[r] & 0xFFFFu);
            const float f1 = T::to_float(s.scale[r] >> 16);
#pragma unroll
            for (int mb = 0; mb < MB; ++mb) {
              acc[r][mb][0] = fmaf(f0, dd[mb][0], acc[r][mb][0]);
              acc[r][mb][1] = fmaf(f0, dd[mb][1], acc[r][mb][1]);
              acc[r][mb][2] = fmaf(f1, dd[mb][2], acc[r][mb][2]);
              acc[r][mb][3] = fmaf(f1, dd[mb][3], acc[r][mb][3]);
            }
          }
        }
        if (j + kDepth < mine) load_w(s, j + kDepth);
      }
    }
  }

  // ---------------------------------------------------------------- reduction over warps
#pragma unroll
  for (int r = 0; r < RT; ++r)
#pragma unroll
    for (int mb = 0; mb < MB; ++mb)
#pragma unroll
      for (int c = 0; c < 4; ++c) red[(warp * kVals + (r * MB + mb) * 4 + c) * 32 + lane] = acc[r][mb][c];
  if (threadIdx.x == 0) bad = !hdr_ok;
  __syncthreads();
  if (bad) {
    if (threadIdx.x == 0) atomicOr(err, 1);
    return;
  }
  for (int e = threadIdx.x; e < kVals * 32; e += blockDim.x) {
    const int ln = e % 32, vi = e / 32;
    float v = 0.f;
    for (int w = 0; w < W; ++w) v += red[(w * kVals + vi) * 32 + ln];
    const int c = vi % 4, mb = (vi / 4) % MB, r = vi / (4 * MB);
    const int row = 16 * (i0 + r) + (ln >> 2) + 8 * (c >> 1);
    const int m = m0 + 8 * mb + 2 * (ln & 3) + (c & 1);
    const int n = b * kBlockN + row;
    if (m < M && n < N && in_extent(y + (size_t)m * N + n, 2, y, yext, err)) y[(size_t)m * N + n] = T::from_float(v);
  }
}


// ---------------------------------------------------------------------------------------------
// Lean variant for M <= 8 (the decode case): a warp streams its x slices into a private
// shared-memory ring with cp.async, issued together with the weights D chunks ahead, so x costs
// no registers and the kernel fits in <= 64 registers per thread -- four 8-warp CTAs per SM.
// HBM throughput of plain loads follows the number of warps with loads outstanding more than
// the bytes each has in flight, so this is what lets the decode stream reach the bandwidth.
constexpr int kSmallRows = 8;   // rows of x per CTA in the lean variant: the 8 columns of the MMA's B
constexpr int kSmallWarps = 8;

// The x ring's layout.  A slot holds rows m < 8 of 128 k, 256 bytes a row, as 16 pieces of 8 k.
// With SW (more than 4 rows of x), piece q of row m sits at q ^ (2 ((q >> 3) & 1) | (m & 1)): a
// quarter-warp's reads (rows r8 of one parity pair, spans t = 0..3, one 8-k step) then hit 8
// different 16-byte bank groups, where the plain layout puts all rows, and the spans t and t + 2,
// on the same ones (measured: the 131072-column head at M = 8 took 33 us swizzled against 42).
// With few rows the plain layout is kept: fewer lanes read, and the XOR costs issue slots in a
// conversion that is issue-bound (the M = 1 step lost 12% with it).
template <bool SW>
__device__ __forceinline__ int xring_piece(int m, int q) {
  return SW ? (q ^ ((2 * ((q >> 3) & 1)) | (m & 1))) : q;
}

// One chunk slot of a lean or streaming CTA: (q - z) * s * x of the lane's weights (RT row-tiles x
// rows r8, r8 + 8 x its 32 k) into the MMA accumulators acc[RT][4]; xs: the lane's 32 k of x row
// r8 in shared memory (zeros where xrow is false), its 8-k step w at byte 16 w, or (16 w) ^ xc
// in the swizzled layout.
template <class T, int RT, bool FACTOR, bool SW>
__device__ __forceinline__ void slot_mma(const uint4 (&code)[RT][2], const uint32_t (&scale)[RT],
                                         const uint32_t (&zero)[RT], const uint8_t *xs, int xc, bool xrow,
                                         float (&acc)[RT][4]) {
#pragma unroll
  for (int r = 0; r < RT; ++r) {
    const ZeroBias zb0 = T::zb(zero[r] & 0xFu), zb1 = T::zb((zero[r] >> 4) & 0xFu);
    float dd[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const uint4 c0 = code[r][0], c1 = code[r][1];
      const uint32_t w0 = (w == 0) ? c0.x : (w == 1) ? c0.y : (w == 2) ? c0.z : c0.w;
      const uint32_t w1 = (w == 0) ? c1.x : (w == 1) ? c1.y : (w == 2) ? c1.z : c1.w;
      uint32_t v0[4], v1[4];
      T::qz(w0, zb0, v0);
      T::qz(w1, zb1, v1);
      if (!FACTOR) {
        const uint32_t s20 = (scale[r] & 0xFFFFu) * 0x00010001u, s21 = (scale[r] >> 16) * 0x00010001u;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          v0[e] = T::mul2(v0[e], s20);
          v1[e] = T::mul2(v1[e], s21);
        }
      }
      const uint4 xw = xrow ? *reinterpret_cast<const uint4 *>(xs + (SW ? ((16 * w) ^ xc) : 16 * w))
                            : make_uint4(0, 0, 0, 0);
      float *dst = FACTOR ? dd : acc[r];
      T::mma16816(dst, v0[0], v1[0], v0[1], v1[1], xw.x, xw.y);  // k 8w + 0..3
      T::mma16816(dst, v0[2], v1[2], v0[3], v1[3], xw.z, xw.w);  // k 8w + 4..7
    }
    if (FACTOR) {
      const float f0 = T::to_float(scale[r] & 0xFFFFu);
      const float f1 = T::to_float(scale[r] >> 16);
      acc[r][0] = fmaf(f0, dd[0], acc[r][0]);
      acc[r][1] = fmaf(f0, dd[1], acc[r][1]);
      acc[r][2] = fmaf(f1, dd[2], acc[r][2]);
      acc[r][3] = fmaf(f1, dd[3], acc[r][3]);
    }
  }
}

template <class T, int D, int RT, bool FACTOR, bool SW>
__global__ void __launch_bounds__(kSmallWarps * 32, RT == 1 ? 4 : 3) gemv_small_kernel(
    const uint16_t *__restrict__ x, const uint8_t *__restrict__ packed, int M, int N, int K, int g, int KT,
    uint16_t *__restrict__ y, int *err) {
  // x ring: [warp][D slots][kSmallRows rows][128 k] fp16 = 2 KB per slot
  __shared__ __align__(16) uint8_t xring[kSmallWarps][D][kSmallRows * 256];
  __shared__ float red[kSmallWarps][RT * 4][32];
  __shared__ int bad;

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int r8 = lane >> 2, t = lane & 3;
  const int tile0 = blockIdx.x * RT;  // RT row-tiles of one n-block (tiles come in fours)
  const int b = tile0 / 4, i0 = tile0 % 4;
  const int CB = chunk_bytes(g);
  const uint8_t *body = packed + kHeaderBytes + (size_t)b * KT * CB;
  const int mine = (KT - warp + kSmallWarps - 1) / kSmallWarps;  // chunks warp, warp + 8, ...

  const long long pext = packed_extent(K, N, g), xext = 2LL * M * K, yext = 2LL * M * N;
  int hdr_ok = 1;
  if (threadIdx.x == 0) hdr_ok = header_ok<T>(packed, K, N, g, pext, err);  // checked at the end

  uint4 code[D][RT][2];
  uint32_t scale[D][RT], zero[D][RT];
  auto load_w = [&](int d, int j) {
    const uint8_t *ch = body + (size_t)(warp + j * kSmallWarps) * CB;
    const uint8_t *meta = ch + kCodeBytes + ((32 * t) / g) * kGroupMetaBytes;
#pragma unroll
    for (int r = 0; r < RT; ++r) {
      const int i = i0 + r;
#pragma unroll
      for (int h = 0; h < 2; ++h)
        code[d][r][h] = ld_w16(ch + (16 * i + r8 + 8 * h) * kRowBytes + 16 * t, packed, pext, err);
      scale[d][r] = ld_w4(meta + 2 * (8 * r8 + 2 * i), packed, pext, err);
      zero[d][r] = ld_w1(meta + kScaleBytes + 4 * r8 + i, packed, pext, err);
    }
  };
  // x rows 0..M-1 of chunk j into slot d: M * 16 pieces of 16 bytes, lane p takes pieces p, p+32..
  auto load_x = [&](int d, int j) {
    const int k0 = (warp + j * kSmallWarps) * kTileK;
    for (int p = lane; p < M * 16; p += 32) {
      const int m = p / 16, q = p % 16;
      const bool ok = k0 + 8 * q < K && in_extent(x + (size_t)m * K + k0 + 8 * q, 16, x, xext, err);
      cp_async16_zfill(&xring[warp][d][m * 256 + 16 * xring_piece<SW>(m, q)], ok ? x + (size_t)m * K + k0 + 8 * q : x,
                       ok);
    }
  };
  const int xc = 16 * ((2 * (t >> 1)) | (r8 & 1));  // this lane's swizzle of its 16-byte reads

  float acc[RT][4];
#pragma unroll
  for (int r = 0; r < RT; ++r)
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[r][c] = 0.f;
#pragma unroll
  for (int d = 0; d < D; ++d)
    if (d < mine) load_w(d, d);
  griddep_launch_dependents();
  griddep_wait();  // x may be the previous kernel's output; y may still be read by it
#pragma unroll
  for (int d = 0; d < D; ++d) {
    if (d < mine) load_x(d, d);
    cp_async_commit();  // one group per slot, possibly empty
  }

#pragma unroll 1
  for (int j0 = 0; j0 < mine; j0 += D) {
#pragma unroll
    for (int d = 0; d < D; ++d) {
      const int j = j0 + d;
      if (j < mine) {
        cp_async_wait_pending<D - 1>();  // this slot's x has landed (for this lane's pieces)
        __syncwarp();                     // ... and every lane's pieces are visible
        slot_mma<T, RT, FACTOR, SW>(code[d], scale[d], zero[d], &xring[warp][d][r8 * 256 + 64 * t], xc, r8 < M, acc);
        __syncwarp();  // every lane is done reading the slot before it is refilled
        if (j + D < mine) {
          load_w(d, j + D);
          load_x(d, j + D);
        }
        cp_async_commit();
      }
    }
  }

#pragma unroll
  for (int r = 0; r < RT; ++r)
#pragma unroll
    for (int c = 0; c < 4; ++c) red[warp][4 * r + c][lane] = acc[r][c];
  if (threadIdx.x == 0) bad = !hdr_ok;
  __syncthreads();
  if (bad) {
    if (threadIdx.x == 0) atomicOr(err, 1);
    return;
  }
  if (threadIdx.x < RT * 128) {
    const int ln = threadIdx.x % 32, c = (threadIdx.x / 32) % 4, r = threadIdx.x / 128;
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < kSmallWarps; ++w) v += red[w][4 * r + c][ln];
    const int row = 16 * (i0 + r) + (ln >> 2) + 8 * (c >> 1);
    const int m = 2 * (ln & 3) + (c & 1);
    const int n = b * kBlockN + row;
    if (m < M && n < N && in_extent(y + (size_t)m * N + n, 2, y, yext, err)) y[(size_t)m * N + n] = T::from_float(v);
  }
}


// ---------------------------------------------------------------------------------------------
// Streaming variant for very wide layers with K <= 2048 (at most two chunks per warp), where the
// lean kernel would need more than two waves of CTAs (the tied LM head: 8192 row-tiles).  Three
// CTAs per SM stay resident and walk pairs of row-tiles u = blockIdx.x, + gridDim.x, ...; x is
// fetched once into shared memory; a warp requests its weights of the next pair as soon as those
// of the current pair are in registers, so the weight stream does not wait for a CTA to exit and
// a new one to start.  The cross-warp sums alternate between two shared buffers, so a pair costs
// one barrier (measured: the LM head at M = 1 31.7 -> 31.25 us against two barriers per pair).
// The packed header is checked before any weight is read.
template <class T, bool FACTOR, bool SW>
__global__ void __launch_bounds__(kSmallWarps * 32, 3) gemv_stream_kernel(
    const uint16_t *__restrict__ x, const uint8_t *__restrict__ packed, int M, int N, int K, int g, int KT,
    int units, uint16_t *__restrict__ y, int *err) {
  constexpr int RT = 2, D = 2;
  __shared__ __align__(16) uint8_t xring[kSmallWarps][D][kSmallRows * 256];
  __shared__ float red[2][kSmallWarps][RT * 4][32];  // alternate buffers: one barrier per pair
  __shared__ int bad;

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int r8 = lane >> 2, t = lane & 3;
  const int CB = chunk_bytes(g);
  const int mine = (KT - warp + kSmallWarps - 1) / kSmallWarps;  // chunks warp, warp + 8 (KT <= 16)

  const long long pext = packed_extent(K, N, g), xext = 2LL * M * K, yext = 2LL * M * N;
  if (threadIdx.x == 0) {
    bad = !header_ok<T>(packed, K, N, g, pext, err);
    if (bad && blockIdx.x == 0) atomicOr(err, 1);
  }
  __syncthreads();
  if (bad) return;

  uint4 code[D][RT][2];
  uint32_t scale[D][RT], zero[D][RT];
  auto load_w = [&](int d, int u) {  // chunk warp + 8 d of row-tile pair u
    const int tile0 = u * RT, b = tile0 / 4, i0 = tile0 % 4;
    const uint8_t *ch = packed + kHeaderBytes + ((size_t)b * KT + warp + d * kSmallWarps) * CB;
    const uint8_t *meta = ch + kCodeBytes + ((32 * t) / g) * kGroupMetaBytes;
#pragma unroll
    for (int r = 0; r < RT; ++r) {
      const int i = i0 + r;
#pragma unroll
      for (int h = 0; h < 2; ++h)
        code[d][r][h] = ld_w16(ch + (16 * i + r8 + 8 * h) * kRowBytes + 16 * t, packed, pext, err);
      scale[d][r] = ld_w4(meta + 2 * (8 * r8 + 2 * i), packed, pext, err);
      zero[d][r] = ld_w1(meta + kScaleBytes + 4 * r8 + i, packed, pext, err);
    }
  };

  int u = blockIdx.x;
#pragma unroll
  for (int d = 0; d < D; ++d)
    if (d < mine) load_w(d, u);
  griddep_launch_dependents();
  griddep_wait();  // x may be the previous kernel's output; y may still be read by it
#pragma unroll
  for (int d = 0; d < D; ++d) {
    if (d < mine) {
      const int k0 = (warp + d * kSmallWarps) * kTileK;
      for (int pp = lane; pp < M * 16; pp += 32) {
        const int m = pp / 16, q = pp % 16;
        const bool ok = k0 + 8 * q < K && in_extent(x + (size_t)m * K + k0 + 8 * q, 16, x, xext, err);
        cp_async16_zfill(&xring[warp][d][m * 256 + 16 * xring_piece<SW>(m, q)],
                         ok ? x + (size_t)m * K + k0 + 8 * q : x, ok);
      }
    }
  }
  const int xc = 16 * ((2 * (t >> 1)) | (r8 & 1));
  cp_async_commit();
  cp_async_wait_pending<0>();
  __syncwarp();

  for (int it = 0; u < units; u += gridDim.x, ++it) {
    float (*rb)[RT * 4][32] = red[it & 1];
    float acc[RT][4];
#pragma unroll
    for (int r = 0; r < RT; ++r)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[r][c] = 0.f;
    const int un = u + (int)gridDim.x;
#pragma unroll
    for (int d = 0; d < D; ++d) {
      if (d < mine) {
        slot_mma<T, RT, FACTOR, SW>(code[d], scale[d], zero[d], &xring[warp][d][r8 * 256 + 64 * t], xc, r8 < M, acc);
        if (un < units) load_w(d, un);  // the next pair's weights stream in meanwhile
      }
    }
#pragma unroll
    for (int r = 0; r < RT; ++r)
#pragma unroll
      for (int c = 0; c < 4; ++c) rb[warp][4 * r + c][lane] = acc[r][c];
    __syncthreads();  // also: every thread is done reading this buffer two pairs ago
    if (threadIdx.x < RT * 128) {
      const int ln = threadIdx.x % 32, c = (threadIdx.x / 32) % 4, r = threadIdx.x / 128;
      float v = 0.f;
#pragma unroll
      for (int w = 0; w < kSmallWarps; ++w) v += rb[w][4 * r + c][ln];
      const int tile0 = u * RT, b = tile0 / 4, i0 = tile0 % 4;
      const int row = 16 * (i0 + r) + (ln >> 2) + 8 * (c >> 1);
      const int m = 2 * (ln & 3) + (c & 1);
      const int n = b * kBlockN + row;
      if (m < M && n < N && in_extent(y + (size_t)m * N + n, 2, y, yext, err)) y[(size_t)m * N + n] = T::from_float(v);
    }
  }
}

// ---------------------------------------------------------------------------------------------
// Mid-size decode, 17 <= M <= 32 rows of x (MB = 3 up to 24 rows, else 4): one pass over
// the weights, where gemv_kernel would take two 16-row passes, each warp fetching from L2 the x of
// every chunk it takes (four to eight times the bytes of the weights it multiplies).  A CTA owns
// one n-block (64 columns: its 4 warps take one row-tile each) over a range of chunks and stages
// each chunk of x once in a shared-memory ring (cp.async, the swizzled layout of the lean kernel)
// that all four warps read, so x costs twice the weights' bytes.  K is split over the S CTAs of
// a thread-block cluster (grid: n-blocks x S); each leaves its fp32 partial in shared memory and
// adds 1/S of the n-block's outputs over the S partials in rank order (its own from its shared
// memory, the others' through distributed shared memory), so y does not depend on timing.
constexpr int kMidWarps = 4;      // one per row-tile of the n-block
constexpr int kMidDepth = 4;      // chunks of weights in flight per warp (registers)
constexpr int kMidSlots = 4;      // chunks of x staged in shared memory; equal to kMidDepth
constexpr int kMidMaxSplits = 8;  // portable cluster size

template <class T, int MB, bool FACTOR>
__global__ void __launch_bounds__(32 * kMidWarps) gemv_mid_kernel(const uint16_t *__restrict__ x,
                                                                 const uint8_t *__restrict__ packed, int M, int N,
                                                                 int K, int g, int KT, int cps, int S,
                                                                 uint16_t *__restrict__ y, int *err) {
  constexpr int R = 8 * MB;             // rows of x per slot (zeros past M)
  constexpr int kSlotBytes = R * 256;   // 128 k of fp16 per row
  constexpr int kVals = MB * 4;         // accumulator values per lane
  static_assert(kMidWarps * kVals * 32 * 4 <= kMidSlots * kSlotBytes, "partials fit in the x ring");
  __shared__ __align__(16) uint8_t xs[kMidSlots * kSlotBytes];
  __shared__ int bad;

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int r8 = lane >> 2, t = lane & 3;
  const int b = blockIdx.x, z = blockIdx.y;  // n-block; split = rank in the cluster
  const int c0 = z * cps, nch = max(0, min(KT, c0 + cps) - c0);
  const int CB = chunk_bytes(g);
  const uint8_t *body = packed + kHeaderBytes + ((size_t)b * KT + c0) * CB;
  const long long pext = packed_extent(K, N, g), xext = 2LL * M * K, yext = 2LL * M * N;
  int hdr_ok = 1;
  if (threadIdx.x == 0) hdr_ok = header_ok<T>(packed, K, N, g, pext, err);

  auto load_w = [&](Stage<1> &st, int j) {  // chunk c0 + j of row-tile `warp`
    const uint8_t *ch = body + (size_t)j * CB;
    const uint8_t *meta = ch + kCodeBytes + ((32 * t) / g) * kGroupMetaBytes;
#pragma unroll
    for (int h = 0; h < 2; ++h) st.code[0][h] = ld_w16(ch + (16 * warp + r8 + 8 * h) * kRowBytes + 16 * t, packed, pext, err);
    st.scale[0] = ld_w4(meta + 2 * (8 * r8 + 2 * warp), packed, pext, err);
    st.zero[0] = ld_w1(meta + kScaleBytes + 4 * r8 + warp, packed, pext, err);
  };
  // x rows 0..R-1 of chunk c0 + j into slot `slot`, by all threads (16-byte pieces)
  auto load_x = [&](int slot, int j) {
    const int k0 = (c0 + j) * kTileK;
    uint8_t *dst = xs + slot * kSlotBytes;
#pragma unroll
    for (int i = 0; i < MB; ++i) {
      const int p = (int)threadIdx.x + i * 32 * kMidWarps, m = p >> 4, q = p & 15;
      const bool ok = m < M && k0 + 8 * q < K && in_extent(x + (size_t)m * K + k0 + 8 * q, 16, x, xext, err);
      cp_async16_zfill(dst + m * 256 + 16 * xring_piece<true>(m, q), ok ? x + (size_t)m * K + k0 + 8 * q : x, ok);
    }
  };

  Stage<1> st[kMidDepth];
#pragma unroll
  for (int d = 0; d < kMidDepth; ++d)
    if (d < nch) load_w(st[d], d);
  griddep_launch_dependents();
  griddep_wait();  // x may be the previous kernel's output; y may still be read by it
#pragma unroll
  for (int d = 0; d < kMidSlots - 1; ++d) {
    if (d < nch) load_x(d, d);
    cp_async_commit();  // one group per chunk, possibly empty
  }

  float acc[MB][4];
#pragma unroll
  for (int mb = 0; mb < MB; ++mb)
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[mb][c] = 0.f;
  const int xc = 16 * ((2 * (t >> 1)) | (r8 & 1));  // the lane's reads in the swizzled slot

#pragma unroll 1
  for (int j0 = 0; j0 < nch; j0 += kMidDepth) {
#pragma unroll
    for (int d = 0; d < kMidDepth; ++d) {
      const int j = j0 + d;  // uniform over the CTA
      if (j < nch) {
        cp_async_wait_pending<kMidSlots - 2>();  // chunk j's x has landed (this thread's pieces)
        __syncthreads();                          // ... every thread's; slot (j - 1) % kMidSlots is free
        if (j + kMidSlots - 1 < nch) load_x((d + kMidSlots - 1) % kMidSlots, j + kMidSlots - 1);
        cp_async_commit();
        const uint8_t *xsl = xs + d * kSlotBytes + 64 * t;  // slot j % kMidSlots == d
        Stage<1> &s = st[d];
        const ZeroBias zb0 = T::zb(s.zero[0] & 0xFu), zb1 = T::zb((s.zero[0] >> 4) & 0xFu);
        float dd[MB][4];
#pragma unroll
        for (int mb = 0; mb < MB; ++mb)
#pragma unroll
          for (int e = 0; e < 4; ++e) dd[mb][e] = 0.f;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const uint32_t w0 = (w == 0) ? s.code[0][0].x : (w == 1) ? s.code[0][0].y : (w == 2) ? s.code[0][0].z : s.code[0][0].w;
          const uint32_t w1 = (w == 0) ? s.code[0][1].x : (w == 1) ? s.code[0][1].y : (w == 2) ? s.code[0][1].z : s.code[0][1].w;
          uint32_t v0[4], v1[4];
          T::qz(w0, zb0, v0);
          T::qz(w1, zb1, v1);
          if (!FACTOR) {
            const uint32_t s20 = (s.scale[0] & 0xFFFFu) * 0x00010001u, s21 = (s.scale[0] >> 16) * 0x00010001u;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              v0[e] = T::mul2(v0[e], s20);
              v1[e] = T::mul2(v1[e], s21);
            }
          }
#pragma unroll
          for (int mb = 0; mb < MB; ++mb) {
            float *dst = FACTOR ? dd[mb] : acc[mb];
            const uint4 xw = *reinterpret_cast<const uint4 *>(xsl + (8 * mb + r8) * 256 + ((16 * w) ^ xc));
            T::mma16816(dst, v0[0], v1[0], v0[1], v1[1], xw.x, xw.y);  // k 8w + 0..3
            T::mma16816(dst, v0[2], v1[2], v0[3], v1[3], xw.z, xw.w);  // k 8w + 4..7
          }
        }
        if (FACTOR) {
          const float f0 = T::to_float(s.scale[0] & 0xFFFFu);
          const float f1 = T::to_float(s.scale[0] >> 16);
#pragma unroll
          for (int mb = 0; mb < MB; ++mb) {
            acc[mb][0] = fmaf(f0, dd[mb][0], acc[mb][0]);
            acc[mb][1] = fmaf(f0, dd[mb][1], acc[mb][1]);
            acc[mb][2] = fmaf(f1, dd[mb][2], acc[mb][2]);
            acc[mb][3] = fmaf(f1, dd[mb][3], acc[mb][3]);
          }
        }
        if (j + kMidDepth < nch) load_w(s, j + kMidDepth);
      }
    }
  }

  // ---------------------------------------------------------------- reduction over the cluster
  cp_async_wait_pending<0>();
  __syncthreads();  // every warp is done with the x ring: it now holds the partials
  float *red = reinterpret_cast<float *>(xs);  // [warp][kVals][32]
#pragma unroll
  for (int mb = 0; mb < MB; ++mb)
#pragma unroll
    for (int c = 0; c < 4; ++c) red[(warp * kVals + mb * 4 + c) * 32 + lane] = acc[mb][c];
  if (threadIdx.x == 0) bad = !hdr_ok;  // the same verdict in every CTA: one packed buffer
  if (S > 1) {
    cluster_arrive();  // release: the partials are visible to the cluster
    cluster_wait();
  } else {
    __syncthreads();
  }
  if (bad) {
    if (z == 0 && threadIdx.x == 0) atomicOr(err, 1);
  } else {
    constexpr int E = kMidWarps * kVals * 32;
    const int e1 = (z + 1) * E / S;
    for (int e = z * E / S + (int)threadIdx.x; e < e1; e += 32 * kMidWarps) {
      float v = 0.f;
      for (int zz = 0; zz < S; ++zz) v += zz == z ? red[e] : ld_cluster_f32(mapa_shared(red + e, (uint32_t)zz));
      const int ln = e & 31, vi = (e >> 5) % kVals, wp = e / (32 * kVals);
      const int c = vi & 3, mb = vi >> 2;
      const int n = b * kBlockN + 16 * wp + (ln >> 2) + 8 * (c >> 1);
      const int m = 8 * mb + 2 * (ln & 3) + (c & 1);
      if (m < M && n < N && in_extent(y + (size_t)m * N + n, 2, y, yext, err)) y[(size_t)m * N + n] = T::from_float(v);
    }
  }
  if (S > 1) {
    cluster_arrive();  // no CTA leaves while another still reads its partials
    cluster_wait();
  }
}

int sm_count() {
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

template <class T, int RT, int MB, bool FACTOR>
cudaError_t launch_variant(int tiles, int mblocks, int W, const uint16_t *x, const uint8_t *packed, int M, int N,
                           int K, int g, int KT, uint16_t *y, int *err, cudaStream_t stream) {
  const int smem = W * RT * MB * 4 * 32 * 4;
  static std::atomic<bool> configured[64];  // per device: the attribute has been set
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !configured[dev].load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(gemv_kernel<T, RT, MB, FACTOR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         160 * 1024);
    if (e != cudaSuccess) return e;
    configured[dev].store(true, std::memory_order_release);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((tiles + RT - 1) / RT, mblocks);
  cfg.blockDim = dim3(32 * W);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemv_kernel<T, RT, MB, FACTOR>, x, packed, M, N, K, g, KT, y, err);
}

template <class T, int RT>
cudaError_t launch_rt(int tiles, int W, int MB, bool factor, const uint16_t *x, const uint8_t *p, int M, int N,
                      int K, int g, int KT, uint16_t *y, int *err, cudaStream_t stream) {
  if (MB == 1)
    return factor ? launch_variant<T, RT, 1, true>(tiles, 1, W, x, p, M, N, K, g, KT, y, err, stream)
                  : launch_variant<T, RT, 1, false>(tiles, 1, W, x, p, M, N, K, g, KT, y, err, stream);
  return factor ? launch_variant<T, RT, 2, true>(tiles, 1, W, x, p, M, N, K, g, KT, y, err, stream)
                : launch_variant<T, RT, 2, false>(tiles, 1, W, x, p, M, N, K, g, KT, y, err, stream);
}

template <class T>
cudaError_t launch_stream(int tiles, bool factor, const uint16_t *x, const uint8_t *p, int M, int N, int K, int g,
                          int KT, uint16_t *y, int *err, cudaStream_t stream) {
  const int units = (tiles + 1) / 2;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(std::min(units, 3 * sm_count()));
  cfg.blockDim = dim3(32 * kSmallWarps);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (M > 4)
    return factor ? cudaLaunchKernelEx(&cfg, gemv_stream_kernel<T, true, true>, x, p, M, N, K, g, KT, units, y, err)
                  : cudaLaunchKernelEx(&cfg, gemv_stream_kernel<T, false, true>, x, p, M, N, K, g, KT, units, y, err);
  return factor ? cudaLaunchKernelEx(&cfg, gemv_stream_kernel<T, true, false>, x, p, M, N, K, g, KT, units, y, err)
                : cudaLaunchKernelEx(&cfg, gemv_stream_kernel<T, false, false>, x, p, M, N, K, g, KT, units, y, err);
}

// Dynamic shared memory (unused) that caps a lean CTA at two per SM: more than a third of the
// SM's shared memory, with the CTA's static shared memory and the per-CTA reservation counted.
template <class T, int D, int RT, bool FACTOR, bool SW>
size_t two_per_sm_pad() {
  auto kernel = gemv_small_kernel<T, D, RT, FACTOR, SW>;
  static std::atomic<long long> pad[64];  // per kernel and device, 0 until computed (stored + 1)
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return 0;
  long long v = pad[dev].load(std::memory_order_relaxed);
  if (!v) {
    int per_sm = 0, reserved = 0;
    cudaFuncAttributes fa = {};
    cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev);
    long long need = 0;
    if (per_sm > 0 && cudaFuncGetAttributes(&fa, kernel) == cudaSuccess) {
      need = per_sm / 3 + 1024 - (long long)fa.sharedSizeBytes - reserved;
      need = need < 0 ? 0 : ((need + 1023) / 1024) * 1024;
      // static + dynamic above 48 KB needs the opt-in; without it, leave the grid as it is
      if (need > 0 && cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)need) != cudaSuccess) {
        cudaGetLastError();
        need = 0;
      }
    }
    v = need + 1;
    pad[dev].store(v, std::memory_order_relaxed);
  }
  return (size_t)(v - 1);
}

template <class T, int D, int RT>
cudaError_t launch_small(int tiles, bool factor, const uint16_t *x, const uint8_t *p, int M, int N, int K, int g,
                         int KT, uint16_t *y, int *err, cudaStream_t stream, bool spread = false) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((tiles + RT - 1) / RT);
  cfg.blockDim = dim3(32 * kSmallWarps);
  // swizzled x ring: measured faster at M = 8 (gate_up 6.14 -> 6.0 us) but slower at M = 5
  // (q_k_v 2.82 -> 3.07 us) in this kernel; the streaming kernel takes it from M = 5
  const bool sw = M >= 8;
  cfg.dynamicSmemBytes = !spread ? 0
                         : factor ? (sw ? two_per_sm_pad<T, D, RT, true, true>() : two_per_sm_pad<T, D, RT, true, false>())
                                  : (sw ? two_per_sm_pad<T, D, RT, false, true>() : two_per_sm_pad<T, D, RT, false, false>());
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (sw)
    return factor ? cudaLaunchKernelEx(&cfg, gemv_small_kernel<T, D, RT, true, true>, x, p, M, N, K, g, KT, y, err)
                  : cudaLaunchKernelEx(&cfg, gemv_small_kernel<T, D, RT, false, true>, x, p, M, N, K, g, KT, y, err);
  return factor ? cudaLaunchKernelEx(&cfg, gemv_small_kernel<T, D, RT, true, false>, x, p, M, N, K, g, KT, y, err)
                : cudaLaunchKernelEx(&cfg, gemv_small_kernel<T, D, RT, false, false>, x, p, M, N, K, g, KT, y, err);
}

// Dynamic shared memory (unused) that holds a mid-size kernel to `per` CTAs per SM: more than
// 1 / (per + 1) of the SM's shared memory with the static part and the per-CTA reservation.
// The kernel's opt-in limit is set once, to the largest pad (per = 1), and never lowered, so
// every pad stays launchable whatever order the launches come in (cached per kernel and device).
template <class T, int MB, bool FACTOR>
size_t mid_pad(int per) {
  auto kernel = gemv_mid_kernel<T, MB, FACTOR>;
  static std::atomic<int> state[64];  // 0: not looked up; 1: ready; -1: no pads
  static std::atomic<long long> per_sm[64], fixed[64];  // shared memory per SM; static part + reservation
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || per < 1) return 0;
  int st = state[dev].load(std::memory_order_acquire);
  if (!st) {
    int sm = 0, reserved = 0;
    cudaFuncAttributes fa = {};
    cudaDeviceGetAttribute(&sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev);
    st = -1;
    if (sm > 0 && cudaFuncGetAttributes(&fa, kernel) == cudaSuccess) {
      const long long fx = (long long)fa.sharedSizeBytes + reserved;
      per_sm[dev].store(sm, std::memory_order_relaxed);
      fixed[dev].store(fx, std::memory_order_relaxed);
      const long long largest = ((sm / 2 + 1024 - fx + 1023) / 1024) * 1024;
      if (largest > 0 && cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)largest) == cudaSuccess)
        st = 1;
    }
    cudaGetLastError();
    state[dev].store(st, std::memory_order_release);
  }
  if (st < 0) return 0;
  const long long need = per_sm[dev].load(std::memory_order_relaxed) / (per + 1) + 1024 -
                         fixed[dev].load(std::memory_order_relaxed);
  return need <= 0 ? 0 : (size_t)(((need + 1023) / 1024) * 1024);
}

// How many CTAs of a mid-size kernel fit per SM, and whether `nclusters` clusters of S of them,
// held to `per` per SM, can be resident at once (cached per kernel, device, S and `per`).
template <class T, int MB, bool FACTOR>
int mid_fit(int S, int nclusters, int per = 0) {
  auto kernel = gemv_mid_kernel<T, MB, FACTOR>;
  static std::atomic<int> per_sm[64];                   // 0 until looked up, else value + 1
  static std::atomic<int> clusters[64][kMidMaxSplits + 1][8];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || S < 1 || S > kMidMaxSplits || per < 0 || per >= 8) return 0;
  if (nclusters <= 0) {  // the CTAs per SM
    int v = per_sm[dev].load(std::memory_order_relaxed);
    if (!v) {
      int n = 0;
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, 32 * kMidWarps, 0) != cudaSuccess) n = 0;
      cudaGetLastError();
      v = (n > 0 ? n : 1) + 1;
      per_sm[dev].store(v, std::memory_order_relaxed);
    }
    return v - 1;
  }
  int v = clusters[dev][S][per].load(std::memory_order_relaxed);
  if (!v) {
    int n = 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1, S);
    cfg.blockDim = dim3(32 * kMidWarps);
    cfg.dynamicSmemBytes = per > 0 ? mid_pad<T, MB, FACTOR>(per) : 0;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = S;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) n = 0;
    cudaGetLastError();
    v = n + 1;
    clusters[dev][S][per].store(v, std::memory_order_relaxed);
  }
  return (v - 1) >= nclusters ? 1 : 0;
}

// Mid-size decode launch: n-blocks x S splits of K, S the largest count (at most 8, at most the
// chunks) whose CTAs fit in one wave and whose clusters are all resident at once.
template <class T, int MB, bool FACTOR>
cudaError_t launch_mid(const uint16_t *x, const uint8_t *p, int M, int N, int K, int g, int KT, uint16_t *y,
                       int *err, cudaStream_t stream) {
  const int NB = num_nblocks(N);
  const long wave = (long)mid_fit<T, MB, FACTOR>(1, 0) * sm_count();
  int S = (int)std::max(1L, std::min<long>(kMidMaxSplits, wave / NB));
  S = std::min(S, KT);
  int cps = (KT + S - 1) / S;
  S = (KT + cps - 1) / cps;  // no empty split
  // The block scheduler fills an SM before it moves on: hold the CTAs to ceil(CTAs / SMs) per SM
  // with unused dynamic shared memory, so that the grid spreads over all SMs.
  const int fit = mid_fit<T, MB, FACTOR>(1, 0);
  auto held = [&](int s) {
    const int per = (int)(((long)NB * s + sm_count() - 1) / sm_count());
    return per < fit ? per : 0;
  };
  while (S > 1 && !mid_fit<T, MB, FACTOR>(S, NB, held(S))) {
    --S;
    cps = (KT + S - 1) / S;
    S = (KT + cps - 1) / cps;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(NB, S);
  cfg.blockDim = dim3(32 * kMidWarps);
  cfg.dynamicSmemBytes = held(S) > 0 ? mid_pad<T, MB, FACTOR>(held(S)) : 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  int na = 1;
  if (S > 1) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 1;
    attr[1].val.clusterDim.y = S;
    attr[1].val.clusterDim.z = 1;
    na = 2;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, gemv_mid_kernel<T, MB, FACTOR>, x, p, M, N, K, g, KT, cps, S, y, err);
}

template <class T>
cudaError_t launch_gemv_t(const uint16_t *x, const void *packed, int M, int N, int K, int g, uint16_t *y,
                          int *err, cudaStream_t stream) {
  const int KT = num_ktiles(K);
  const uint8_t *p = static_cast<const uint8_t *>(packed);
  const bool factor = (g == kTileK);
  // 17..32 rows: one pass over the weights, x shared by the CTA, K split over a cluster
  // (measured against two 16-row passes of gemv_kernel: q_k_v M = 24 6.14 -> 5.12 us, gate_up
  // M = 32 13.9 -> 12.55 us).  At 9..16 rows gemv_kernel's single pass stays faster (the same
  // kernel with 16 rows: q_k_v 3.6 -> 4.1 us, gate_up 7.7 -> 9.2 us, down 6.9 either way).
  if (M > 24)
    return factor ? launch_mid<T, 4, true>(x, p, M, N, K, g, KT, y, err, stream)
                  : launch_mid<T, 4, false>(x, p, M, N, K, g, KT, y, err, stream);
  if (M > 16)  // 24 rows of x per slot (measured against 32: q_k_v M = 24 5.1 -> 4.6 us, gate_up M = 17 12.4 -> 10.5 us)
    return factor ? launch_mid<T, 3, true>(x, p, M, N, K, g, KT, y, err, stream)
                  : launch_mid<T, 3, false>(x, p, M, N, K, g, KT, y, err, stream);
  const int MB = (M <= 8) ? 1 : 2;
  // Row-tiles of 16 columns that hold at least one column < N (N % 8 == 0).
  const int tiles = (N + 15) / 16;
  const long ctas1 = tiles;
  // Lean variant for M <= 8 unless K is long and the grid is small (then 16 warps per CTA win).
  const bool long_k = KT >= 32 && ctas1 <= sm_count();
  if (M <= kSmallRows && !long_k) {
    // one-tile CTAs (4 per SM) while they fit in one wave; two-tile CTAs (3 per SM) beyond, so
    // that every CTA is resident and has issued all its weight loads when the wait ends; resident
    // streaming CTAs where two-tile CTAs would need more than two waves (K <= 2048)
    // When the grid is at most two CTAs per SM, they are held to two per SM: the block scheduler
    // fills an SM before it moves on, so a grid this small would otherwise sit four deep on a
    // third of the SMs (measured: the 192 CTAs of a 2048 x 3072 layer on 50 of 152 SMs).
    if (ctas1 <= 4L * sm_count())
      return launch_small<T, 2, 1>(tiles, factor, x, p, M, N, K, g, KT, y, err, stream, ctas1 <= 2L * sm_count());
    if (KT <= 2 * kSmallWarps && ctas1 > 12L * sm_count())
      return launch_stream<T>(tiles, factor, x, p, M, N, K, g, KT, y, err, stream);
    return launch_small<T, 2, 2>(tiles, factor, x, p, M, N, K, g, KT, y, err, stream);
  }
  // Two row-tiles per CTA once the grid would cover the GPU several times over (a 2-tile CTA
  // never straddles an n-block: tiles come in fours per n-block and pairs start at even tiles);
  // with 16 rows of x the per-CTA weights are reused twice as often, so earlier.  Four warps on
  // large grids, sixteen when K is long and the grid is at most about one CTA per SM (measured).
  const int sms = sm_count();
  const bool two = ctas1 >= (MB == 1 ? 4L : 1L) * sms;
  const int W = (ctas1 >= 4L * sms) ? 4 : (!two && long_k && MB == 1) ? 16 : 8;
  if (two) return launch_rt<T, 2>(tiles, W, MB, factor, x, p, M, N, K, g, KT, y, err, stream);
  return launch_rt<T, 1>(tiles, W, MB, factor, x, p, M, N, K, g, KT, y, err, stream);
}

}  // namespace

cudaError_t launch_gemv(const uint16_t *x, const void *packed, int M, int N, int K, int g, int dtype, uint16_t *y,
                        int *err, cudaStream_t stream) {
  return dtype == kDtypeBf16 ? launch_gemv_t<Bf16>(x, packed, M, N, K, g, y, err, stream)
                             : launch_gemv_t<Fp16>(x, packed, M, N, K, g, y, err, stream);
}

}  // namespace w4a16
