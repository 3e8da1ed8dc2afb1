// dq.cuh -- register-level conversion of packed 4-bit codes to fp16 (device only).
//
// A code word holds 8 consecutive k of one column in slots ordered {0,2,4,6,1,3,5,7}.  OR'ing
// a nibble into the mantissa of fp16 1024.0 (ulp 1) gives 1024 + q exactly; a nibble left in
// bits 4..7 gives 1024 + 16q.  One lop3 per pair of codes therefore yields a half2 of
// consecutive k, and one exact half2 op removes the bias together with the zero point:
//     (1024 + q) - (1024 + z)               = q - z
//     (1024 + 16q) * (1/16) + (-(64 + z))   = q - z          (single rounding of an exact value)
// q - z is a small integer, exact in fp16.  Multiplying by the fp16 scale rounds once, which is
// the layer's fp16 weight fp16((q - z) * s) exactly.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

namespace w4a16 {

__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));  // (a & b) | c
  return d;
}

__device__ __forceinline__ uint32_t h2_as_u32(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }
__device__ __forceinline__ __half2 u32_as_h2(uint32_t u) { return *reinterpret_cast<__half2 *>(&u); }

// Bias constants for zero code z (0..15), both halves equal.
struct ZeroBias {
  uint32_t lo;  // half2(1024 + z)
  uint32_t hi;  // half2(-(64 + z))
};
__device__ __forceinline__ ZeroBias zero_bias(uint32_t z) {
  ZeroBias b;
  b.lo = (0x6400u | z) * 0x00010001u;
  b.hi = (0xD400u | (z << 4)) * 0x00010001u;
  return b;
}

// The four half2 values (q - z) of one code word, in k order: v[0] = (k0, k1), v[1] = (k2, k3),
// v[2] = (k4, k5), v[3] = (k6, k7).
__device__ __forceinline__ void word_to_qz(uint32_t w, ZeroBias zb, uint32_t v[4]) {
  const __half2 sixteenth = u32_as_h2(0x2C002C00u);  // 1/16
  uint32_t w2 = w >> 8;
  v[0] = h2_as_u32(__hsub2(u32_as_h2(lop3_and_or(w, 0x000F000Fu, 0x64006400u)), u32_as_h2(zb.lo)));
  v[1] = h2_as_u32(__hfma2(u32_as_h2(lop3_and_or(w, 0x00F000F0u, 0x64006400u)), sixteenth,
                           u32_as_h2(zb.hi)));
  v[2] = h2_as_u32(__hsub2(u32_as_h2(lop3_and_or(w2, 0x000F000Fu, 0x64006400u)), u32_as_h2(zb.lo)));
  v[3] = h2_as_u32(__hfma2(u32_as_h2(lop3_and_or(w2, 0x00F000F0u, 0x64006400u)), sixteenth,
                           u32_as_h2(zb.hi)));
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
  return h2_as_u32(__hmul2(u32_as_h2(a), u32_as_h2(b)));
}



// ------------------------------------------------------------------------------------------
// bfloat16.  Its 7 fraction bits hold a nibble OR'd into the mantissa of 128.0 (0x4300, ulp 1),
// but not the nibble scaled by 16, so all four pairs of a word come from the low nibble of
// each byte after a shift: (w >> 4i) & 0x000F000F holds slots i and i + 4, i.e. k = 2i, 2i + 1.
// (128 + q) - (128 + z) = q - z is exact, and one bf16 multiply by the scale rounds once.
__device__ __forceinline__ uint32_t bf2_as_u32(__nv_bfloat162 h) { return *reinterpret_cast<uint32_t *>(&h); }
__device__ __forceinline__ __nv_bfloat162 u32_as_bf2(uint32_t u) { return *reinterpret_cast<__nv_bfloat162 *>(&u); }

// Element types of a layer: fp16 (the pages' checkpoints) or bf16 (x, scales and y in bf16).
struct Fp16 {
  static constexpr int kDtype = 0;  // packed header's dtype word
  __device__ static ZeroBias zb(uint32_t z) { return zero_bias(z); }
  __device__ static void qz(uint32_t w, ZeroBias b, uint32_t v[4]) { word_to_qz(w, b, v); }
  __device__ static uint32_t mul2(uint32_t a, uint32_t b) { return hmul2_u32(a, b); }
  __device__ static float to_float(uint32_t bits) { return __half2float(__ushort_as_half((unsigned short)bits)); }
  __device__ static uint16_t from_float(float a) { return __half_as_ushort(__float2half_rn(a)); }
  __device__ static uint32_t pack2(float a, float b) { return h2_as_u32(__floats2half2_rn(a, b)); }
  __device__ static void mma16816(float d[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                  uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
};

struct Bf16 {
  static constexpr int kDtype = 1;
  __device__ static ZeroBias zb(uint32_t z) {
    ZeroBias b;
    b.lo = (0x4300u | z) * 0x00010001u;  // bf16x2(128 + z)
    b.hi = 0;
    return b;
  }
  __device__ static void qz(uint32_t w, ZeroBias b, uint32_t v[4]) {
    const __nv_bfloat162 bias = u32_as_bf2(b.lo);
#pragma unroll
    for (int i = 0; i < 4; ++i)
      v[i] = bf2_as_u32(__hsub2(u32_as_bf2(lop3_and_or(w >> (4 * i), 0x000F000Fu, 0x43004300u)), bias));
  }
  __device__ static uint32_t mul2(uint32_t a, uint32_t b) { return bf2_as_u32(__hmul2(u32_as_bf2(a), u32_as_bf2(b))); }
  __device__ static float to_float(uint32_t bits) { return __uint_as_float(bits << 16); }
  __device__ static uint16_t from_float(float a) { return __bfloat16_as_ushort(__float2bfloat16_rn(a)); }
  __device__ static uint32_t pack2(float a, float b) { return bf2_as_u32(__floats2bfloat162_rn(a, b)); }
  __device__ static void mma16816(float d[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                  uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
};

}  // namespace w4a16
