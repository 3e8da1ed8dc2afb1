// nibble.cuh -- an 8 x 8 transpose of 4-bit codes held in registers, shared by the repack kernel
// (AWQ words -> the packed layout's code words) and the AWQ -> standard converter.
#pragma once

#include <cstdint>

namespace w4a16 {

// Transpose an 8 x 8 matrix of nibbles held as 8 words (row i = R[i], column p = bits 4p..4p+3):
// afterwards R[p] holds, in nibble i, what R[i] held in nibble p.  Three rounds exchange 4-, 8-
// and 16-bit blocks between rows 1, 2 and 4 apart: masked swaps for the nibbles, byte permutes
// for the bytes and half-words.
__device__ __forceinline__ void nibble_transpose8(uint32_t (&R)[8]) {
#pragma unroll
  for (int a = 0; a < 8; a += 2) {
    const uint32_t t = ((R[a] >> 4) ^ R[a + 1]) & 0x0F0F0F0Fu;
    R[a + 1] ^= t;
    R[a] ^= t << 4;
  }
#pragma unroll
  for (int h = 0; h < 4; ++h) {  // rows (0,2) (1,3) (4,6) (5,7): even bytes of a with those of a + 2
    const int a = (h & 1) + 4 * (h >> 1);
    const uint32_t x = R[a], y = R[a + 2];
    R[a] = __byte_perm(x, y, 0x6240);
    R[a + 2] = __byte_perm(x, y, 0x7351);
  }
#pragma unroll
  for (int a = 0; a < 4; ++a) {  // low half-words of a with those of a + 4
    const uint32_t x = R[a], y = R[a + 4];
    R[a] = __byte_perm(x, y, 0x5410);
    R[a + 4] = __byte_perm(x, y, 0x7632);
  }
}

}  // namespace w4a16
